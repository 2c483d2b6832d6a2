"""Pins for the oracle's number formats and quantisers.

Each check compares the oracle against something other than itself: torch's
float8_e4m3fn conversion (a library routine), the published E2M1 value table,
brute-force nearest-value search, or exact arithmetic facts."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _formats():
    with open(os.path.join(GOLD, "formats.json")) as f:
        return json.load(f)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero survives
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0])


def test_e4m3_extremes_match_format_table():
    f = _formats()["e4m3"]
    assert oracle.e4m3_value(f["max_code"]) == f["max_normal"]
    assert oracle.e4m3_value(0x08) == f["min_normal"]
    assert oracle.e4m3_value(0x01) == f["min_subnormal"]
    for c in f["nan_codes"]:
        assert np.isnan(oracle.e4m3_value(c))


def _e4m3_probe_values():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8)).astype(np.float64)
    pos = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (pos[1:] + pos[:-1]) / 2                      # exact ties
    ys = [pos, mids]
    m32 = mids.astype(np.float32)                        # one ulp either side of ties
    ys.append(np.nextafter(m32, np.float32(np.inf), dtype=np.float32))
    ys.append(np.nextafter(m32, np.float32(0), dtype=np.float32))
    rng = np.random.default_rng(7)
    ys.append(np.abs(rng.standard_normal(20000)) * 50)
    ys.append(np.exp(rng.uniform(-12, 6.1, 20000)))
    y = np.concatenate(ys).astype(np.float32)
    y = y[np.abs(y) <= 464.0]                           # torch: NaN from 480 on
    return np.concatenate([y, -y])


def test_e4m3_encode_matches_torch_rne():
    y = _e4m3_probe_values()
    ours = oracle.e4m3_encode(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, (y[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_saturates():
    y = np.array([448.0, 463.9, 464.0, 500.0, 1e6, np.inf, -1e6], np.float32)
    assert list(oracle.e4m3_encode(y)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_e2m1_value_table():
    tab = _formats()["e2m1"]["positive_values_by_code"]
    assert [oracle.e2m1_value(c) for c in range(8)] == tab
    assert [oracle.e2m1_value(8 + c) for c in range(8)] == [-v for v in tab]


def test_e2m1_encode_is_nearest_with_ties_to_even_code():
    tab = np.array(_formats()["e2m1"]["positive_values_by_code"])
    rng = np.random.default_rng(3)
    mids = (tab[1:] + tab[:-1]) / 2
    y = np.concatenate([tab, mids, rng.uniform(0, 8, 5000), [6.5, 7.0, 100.0]]).astype(np.float32)
    y = np.concatenate([y, -y])
    got = oracle.e2m1_encode(y)
    for yi, gi in zip(y, got):
        a = min(abs(float(yi)), 6.0)
        dist = np.abs(tab - a)
        best = np.nonzero(dist == dist.min())[0]
        want = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
        want |= 8 if np.signbit(yi) else 0
        assert gi == want, (yi, gi, want)


def test_quant_e4m3_rows_matches_torch_cast():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    x[5] = 0.0
    x[9] *= 1e-4
    codes, scale = oracle.quant_e4m3_rows(x)
    amax = np.abs(x).max(1)
    assert scale[5] == 1.0 and not codes[5].any()
    nz = amax > 0
    inv = (np.float32(448.0) / amax[nz].astype(np.float32)).astype(np.float32)
    y = (x[nz] * inv[:, None]).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[nz], ref)
    assert np.array_equal(scale[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    # the row maximum always lands on (or next to) the top code
    top = codes[nz][np.arange(nz.sum()), np.abs(x[nz]).argmax(1)] & 0x7F
    assert np.all(top >= 0x7D)


def test_quant_e2m1_blocks_brute_force():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    x[3, :32] = 0.0
    packed, sc = oracle.quant_e2m1_blocks(x)
    tab = np.array(_formats()["e2m1"]["positive_values_by_code"], np.float64)
    for r in range(x.shape[0]):
        for b in range(4):
            blk = x[r, b * 32:(b + 1) * 32]
            amax = np.float32(np.abs(blk).max())
            want_sc = torch.tensor([amax / np.float32(6.0)]).to(torch.float8_e4m3fn).view(torch.uint8).item()
            if want_sc & 0x7F == 0:
                want_sc = 0x01
            assert sc[r, b] == want_sc
            scv = np.float32(oracle.e4m3_value(int(sc[r, b])))
            for c in range(32):
                y = np.float32(blk[c] / scv)
                a = min(abs(float(y)), 6.0)
                dist = np.abs(tab - a)
                best = np.nonzero(dist == dist.min())[0]
                want = best[0] if len(best) == 1 else [i for i in best if i % 2 == 0][0]
                want |= 8 if np.signbit(y) else 0
                byte = packed[r, (b * 32 + c) // 2]
                got = (byte >> 4) if c % 2 else (byte & 0xF)
                assert got == want


def _pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def test_fp4_to_e4m3_lossless_for_power_of_two_scales():
    rng = np.random.default_rng(1)
    rows, d = 32, 128
    codes = rng.integers(0, 16, (rows, d))
    # block scales 2^a with a spread of at most 6 binades: e*sc/S stays on the grid
    sc = np.zeros((rows, 4), np.uint8)
    for r in range(rows):
        top = rng.integers(-3, 6)
        for b in range(4):
            a = top - rng.integers(0, 7)
            sc[r, b] = oracle.e4m3_encode(np.array([2.0 ** a], np.float32))[0]
    x8, S, n_round = oracle.fp4_to_e4m3(_pack(codes), sc)
    assert n_round == 0
    tab = np.array([oracle.e2m1_value(c) for c in range(16)])
    scv = oracle.e4m3_decode(sc).astype(np.float64)
    exact = tab[codes] * np.repeat(scv, 32, axis=1)
    rec = oracle.e4m3_decode(x8).astype(np.float64) * S[:, None]
    assert np.array_equal(rec, exact)
    # S is a power of two placing the largest block scale in [32, 64)
    m = scv.max(1)
    assert np.all((m / S >= 32) & (m / S < 64))
    assert np.all(np.frexp(S)[0] == 0.5)


def test_fp4_to_e4m3_counts_rounding_by_enumeration():
    rng = np.random.default_rng(2)
    rows, d = 24, 128
    codes = rng.integers(0, 16, (rows, d))
    sc = rng.integers(0x30, 0x48, (rows, 4)).astype(np.uint8)   # mantissas vary
    sc[:4] = 0x01            # a row whose spread falls under the subnormal floor
    sc[:4, 0] = 0x60
    x8, S, n_round = oracle.fp4_to_e4m3(_pack(codes), sc)
    grid = oracle.e4m3_decode(np.arange(256, dtype=np.uint8)).astype(np.float64)
    grid = set(grid[np.isfinite(grid)].tolist())
    tab = np.array([oracle.e2m1_value(c) for c in range(16)])
    scv = oracle.e4m3_decode(sc).astype(np.float64)
    y = tab[codes] * np.repeat(scv, 32, axis=1) / S[:, None].astype(np.float64)
    want = sum(1 for v in y.ravel() if float(v) not in grid)
    assert n_round == want and want > 0
    # every element is within half an E4M3 step of the exact product
    rec = oracle.e4m3_decode(x8).astype(np.float64)
    assert np.all(np.abs(rec - y) <= np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) + 1e-12)
