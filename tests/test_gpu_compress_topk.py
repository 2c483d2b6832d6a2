"""GPU parity: compression (with its E4M3 / E2M1 epilogues) and top-k
selection, against the oracle on identical inputs."""
import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import inputs, lib
from helpers import DEV, assert_close, host, sync_status

pytestmark = pytest.mark.gpu


def _compress(x, logits, m, out_dtype):
    B, n, d = x.shape
    Nc = n // m
    xd = lib.F32 if x.dtype == torch.float32 else lib.BF16
    if out_dtype == lib.E4M3:
        out = torch.empty(B, Nc, d, dtype=torch.uint8, device=DEV)
        sc = torch.empty(B, Nc, dtype=torch.float32, device=DEV)
    elif out_dtype == lib.E2M1:
        out = torch.empty(B, Nc, d // 2, dtype=torch.uint8, device=DEV)
        sc = torch.empty(B, Nc, d // 32, dtype=torch.uint8, device=DEV)
    else:
        out = torch.empty(B, Nc, d, dtype=torch.float32 if out_dtype == lib.F32 else torch.bfloat16, device=DEV)
        sc = None
    lib.csa_compress(B, n, m, logits, [x], [xd], [d], [out], [out_dtype], [sc])
    sync_status()
    return out, sc


@pytest.mark.parametrize("m", [1, 4, 128])
@pytest.mark.parametrize("in_dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [32, 128])
def test_compress_float_outputs(m, in_dt, d):
    g = torch.Generator().manual_seed(100 + m + d)
    B, n = 2, m * 37 + (m - 1)            # ragged tail dropped
    x = torch.randn(B, n, d, generator=g).to(in_dt)
    logits = torch.randn(B, n, generator=g) * 2
    want = oracle.compress(logits, x, m)
    for od in (lib.F32, lib.BF16):
        out, _ = _compress(x.to(DEV), logits.to(DEV), m, od)
        got = host(out).float().numpy()
        if od == lib.F32:
            assert_close(got, want, atol=2e-6, rtol=2e-6, what=f"f32 m={m}")
        else:   # one bf16 rounding: half an ulp (2^-8 relative) plus fp32 noise
            assert_close(got, want, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what=f"bf16 m={m}")


def test_compress_multi_stream_shares_logits():
    g = torch.Generator().manual_seed(7)
    B, n, m = 1, 512, 4
    logits = torch.randn(B, n, generator=g)
    xs = [torch.randn(B, n, d, generator=g).to(torch.bfloat16) for d in (128, 64, 128)]
    outs = [torch.empty(B, n // m, x.shape[-1], dtype=torch.bfloat16, device=DEV) for x in xs]
    lib.csa_compress(B, n, m, logits.to(DEV), [x.to(DEV) for x in xs], [lib.BF16] * 3,
                     [x.shape[-1] for x in xs], outs, [lib.BF16] * 3, None)
    sync_status()
    for x, o in zip(xs, outs):
        assert_close(host(o).float().numpy(), oracle.compress(logits, x, m), atol=1e-6, rtol=2.0 ** -8 + 1e-5)


def test_quantisers_bit_exact_on_identity_compression():
    """m = 1 makes the block weight exactly 1, so the compressed value is the
    input itself and the E4M3 / E2M1 codes must match the oracle's bit for bit."""
    g = torch.Generator().manual_seed(11)
    B, n, d = 2, 300, 128
    x = torch.randn(B, n, d, generator=g) * torch.exp(torch.randn(B, n, 1, generator=g) * 2)
    x[0, 5] = 0.0                        # all-zero row -> scale 1
    x[1, 7, :32] = 0.0                   # all-zero FP4 block
    logits = torch.randn(B, n, generator=g)
    codes, scale = _compress(x.to(DEV), logits.to(DEV), 1, lib.E4M3)
    wc, ws = oracle.quant_e4m3_rows(x.numpy())
    assert np.array_equal(host(codes).numpy(), wc)
    assert np.array_equal(host(scale).numpy(), ws)
    packed, sc = _compress(x.to(DEV), logits.to(DEV), 1, lib.E2M1)
    wp, wsc = oracle.quant_e2m1_blocks(x.numpy())
    assert np.array_equal(host(sc).numpy(), wsc)
    assert np.array_equal(host(packed).numpy(), wp)


def test_quantised_compression_within_format_error():
    g = torch.Generator().manual_seed(12)
    B, n, d, m = 1, 4 * 500, 128, 4
    x = torch.randn(B, n, d, generator=g).to(torch.bfloat16)
    logits = torch.randn(B, n, generator=g)
    ref32 = oracle.compress(logits, x, m).astype(np.float32)
    codes, scale = _compress(x.to(DEV), logits.to(DEV), m, lib.E4M3)
    wc, ws = oracle.quant_e4m3_rows(ref32)
    c, s = host(codes).numpy(), host(scale).numpy()
    assert_close(s, ws, atol=0, rtol=1e-6, what="e4m3 scales")
    # codes may differ only where fp32 rounding of the compressed value moves
    # it across a rounding boundary: at most one E4M3 step, and rarely
    dec = oracle.e4m3_decode(c).astype(np.float64) * s[..., None]
    ref = oracle.e4m3_decode(wc).astype(np.float64) * ws[..., None]
    step = np.abs(ref) * 2.0 ** -3 + s[..., None] * 2.0 ** -9 + 1e-12
    assert np.all(np.abs(dec - ref) <= step * 1.0001)
    assert (c != wc).mean() < 1e-3
    packed, sc = _compress(x.to(DEV), logits.to(DEV), m, lib.E2M1)
    wp, wsc = oracle.quant_e2m1_blocks(ref32)
    assert (host(sc).numpy() != wsc).mean() < 1e-3
    assert (host(packed).numpy() != wp).mean() < 2e-3


def _check_e4m3(codes, scale, ref32, what):
    """E4M3 rows against the oracle's quantiser on the fp32-rounded oracle
    compression: scales to 1e-6, codes at most one E4M3 step apart and rarely."""
    wc, ws = oracle.quant_e4m3_rows(ref32)
    c, s = host(codes).numpy(), host(scale).numpy()
    assert_close(s, ws, atol=0, rtol=1e-6, what=f"{what} e4m3 scales")
    dec = oracle.e4m3_decode(c).astype(np.float64) * s[..., None]
    ref = oracle.e4m3_decode(wc).astype(np.float64) * ws[..., None]
    step = np.abs(ref) * 2.0 ** -3 + s[..., None] * 2.0 ** -9 + 1e-12
    assert np.all(np.abs(dec - ref) <= step * 1.0001), what
    assert (c != wc).mean() < 1e-3, what


def _check_e2m1(packed, sc, ref32, what):
    wp, wsc = oracle.quant_e2m1_blocks(ref32)
    assert (host(sc).numpy() != wsc).mean() < 1e-3, what
    assert (host(packed).numpy() != wp).mean() < 2e-3, what


def _alloc_out(B, Nc, d, kind):
    if kind == lib.E4M3:
        return (torch.empty(B, Nc, d, dtype=torch.uint8, device=DEV),
                torch.empty(B, Nc, dtype=torch.float32, device=DEV))
    if kind == lib.E2M1:
        return (torch.empty(B, Nc, d // 2, dtype=torch.uint8, device=DEV),
                torch.empty(B, Nc, d // 32, dtype=torch.uint8, device=DEV))
    dt = torch.float32 if kind == lib.F32 else torch.bfloat16
    return torch.empty(B, Nc, d, dtype=dt, device=DEV), None


def _check_stream(got, sc, want64, kind, what):
    if kind == lib.F32:
        assert_close(host(got).numpy(), want64, atol=2e-6, rtol=2e-6, what=what)
    elif kind == lib.BF16:
        assert_close(host(got).float().numpy(), want64, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what=what)
    elif kind == lib.E4M3:
        _check_e4m3(got, sc, want64.astype(np.float32), what)
    else:
        _check_e2m1(got, sc, want64.astype(np.float32), what)


# Short blocks with m and n multiples of 4 take the tiled all-streams kernel:
# one call mixing input dtypes, widths and every output kind, with a batch of
# two and an entry count that leaves a ragged last tile.
@pytest.mark.parametrize("m", [4, 8, 16, 32])
def test_compress_tiles_mixed_streams(m):
    g = torch.Generator().manual_seed(300 + m)
    B, Nc = 2, 1237
    n = Nc * m + (4 if m > 4 else 0)         # a ragged partial block at the end
    if m < 32:
        spec = [(torch.float32, 64, lib.F32), (torch.bfloat16, 128, lib.BF16),
                (torch.bfloat16, 128, lib.E4M3), (torch.float32, 32, lib.E2M1)]
    else:
        spec = [(torch.bfloat16, 128, lib.BF16), (torch.float32, 32, lib.E2M1)]
    logits = torch.randn(B, n, generator=g) * 2
    xs = [torch.randn(B, n, d, generator=g).to(dt) for dt, d, _ in spec]
    outs = [_alloc_out(B, Nc, d, k) for _, d, k in spec]
    lib.csa_compress(B, n, m, logits.to(DEV), [x.to(DEV) for x in xs],
                     [lib.F32 if dt == torch.float32 else lib.BF16 for dt, _, _ in spec],
                     [d for _, d, _ in spec], [o for o, _ in outs], [k for _, _, k in spec],
                     [sc for _, sc in outs])
    sync_status()
    for (dt, d, kind), x, (o, sc) in zip(spec, xs, outs):
        _check_stream(o, sc, oracle.compress(logits, x, m), kind, f"m={m} d={d} kind={kind}")


def test_compress_tiles_extremes():
    """Closed forms through the tiled kernel: equal logits give the block
    mean; one dominant logit selects its token; a tiny batch of one entry."""
    g = torch.Generator().manual_seed(310)
    B, m, Nc, d = 1, 4, 513, 128
    n = Nc * m
    x = torch.randn(B, n, d, generator=g).to(torch.bfloat16)
    out, _ = _compress(x.to(DEV), torch.zeros(B, n).to(DEV), m, lib.F32)
    mean = x.float().view(B, Nc, m, d).double().mean(2).numpy()
    assert_close(host(out).numpy(), mean, atol=1e-6, rtol=1e-6, what="equal logits -> block mean")
    logits = torch.zeros(B, n)
    pick = torch.randint(0, m, (Nc,), generator=g)
    logits[0, torch.arange(Nc) * m + pick] = 1e4
    out, _ = _compress(x.to(DEV), logits.to(DEV), m, lib.F32)
    sel = x.float().view(B, Nc, m, d)[0, torch.arange(Nc), pick].numpy()[None]
    assert np.array_equal(host(out).numpy(), sel)
    x1 = torch.randn(1, 4, 128, generator=g)
    l1 = torch.randn(1, 4, generator=g)
    out, _ = _compress(x1.to(DEV), l1.to(DEV), 4, lib.F32)
    assert_close(host(out).numpy(), oracle.compress(l1, x1, 4), atol=2e-6, rtol=2e-6, what="one entry")


def test_compress_tiles_stack_size():
    """The hybrid stack's CSA compression at full size: 131,072 tokens, m = 4,
    K and V to BF16 and the indexer key to E2M1, every entry checked."""
    g = torch.Generator().manual_seed(320)
    B, n, m, d = 1, 131072, 4, 128
    logits = torch.randn(B, n, generator=g)
    xs = [torch.randn(B, n, d, generator=g).to(torch.bfloat16) for _ in range(3)]
    kinds = [lib.BF16, lib.BF16, lib.E2M1]
    outs = [_alloc_out(B, n // m, d, k) for k in kinds]
    lib.csa_compress(B, n, m, logits.to(DEV), [x.to(DEV) for x in xs], [lib.BF16] * 3, [d] * 3,
                     [o for o, _ in outs], kinds, [sc for _, sc in outs])
    sync_status()
    for x, kind, (o, sc) in zip(xs, kinds, outs):
        _check_stream(o, sc, oracle.compress(logits, x, m), kind, f"stack kind={kind}")


# ---- top-k on identical scores: bit-exact --------------------------------

def _topk_case(B, n_q, q_pos0, m, Nc, k, tie_levels, seed, order=None, plant_inf=0):
    sc = inputs.random_scores(B * n_q, Nc, seed=seed, tie_levels=tie_levels)
    if plant_inf:   # +inf and -inf at random entries of every row (ties among them go by index)
        g = torch.Generator().manual_seed(seed + 1)
        sc.scatter_(1, torch.randint(0, Nc, (B * n_q, plant_inf), generator=g), float("inf"))
        sc.scatter_(1, torch.randint(0, Nc, (B * n_q, plant_inf), generator=g), float("-inf"))
    if order == "ascending":     # the best entries cluster at the end of the row
        sc = sc.sort(dim=1).values.contiguous()
    elif order == "descending":  # ... or at its start
        sc = sc.sort(dim=1, descending=True).values.contiguous()
    out = torch.empty(B * n_q, k, dtype=torch.int32, device=DEV)
    ws_bytes = lib.csa_topk_select_workspace_size(B, n_q, Nc, k)
    ws = lib.empty_workspace(ws_bytes)
    lib.csa_topk_select(B, n_q, q_pos0, m, Nc, k, sc.to(DEV), out, ws, ws_bytes)
    sync_status()
    t = q_pos0 + np.arange(B * n_q) % n_q
    lens = oracle.visible(t, m, Nc)
    want = oracle.topk(sc.numpy(), lens, k)
    got = host(out).numpy()
    bad = np.nonzero((got != want).any(1))[0]
    assert bad.size == 0, (bad[:5], got[bad[0]][:8], want[bad[0]][:8])


@pytest.mark.parametrize("case", [
    dict(B=1, n_q=70, q_pos0=0, m=4, Nc=300, k=16, tie_levels=0),         # short rows, padding
    dict(B=2, n_q=33, q_pos0=4000, m=4, Nc=5000, k=64, tie_levels=0),
    dict(B=2, n_q=17, q_pos0=4000, m=4, Nc=5000, k=64, tie_levels=3),      # heavy ties
    dict(B=1, n_q=9, q_pos0=32768 * 4 - 5, m=4, Nc=32768, k=1024, tie_levels=0),   # one CTA max
    dict(B=1, n_q=5, q_pos0=160000 - 3, m=4, Nc=40000, k=1024, tie_levels=0),      # two-phase
    dict(B=3, n_q=1, q_pos0=(1 << 20) - 1, m=4, Nc=262144, k=1024, tie_levels=0),   # decode rows
    dict(B=2, n_q=1, q_pos0=(1 << 20) - 1, m=4, Nc=262144, k=1024, tie_levels=50),
    dict(B=1, n_q=3, q_pos0=2000, m=1, Nc=2003, k=4096, tie_levels=0),      # k > row length
    dict(B=2, n_q=1, q_pos0=(1 << 20) - 1, m=4, Nc=262144, k=1024, tie_levels=1),   # threshold bin overflows
    dict(B=1, n_q=4, q_pos0=4 * 33000 - 3, m=4, Nc=33000, k=4096, tie_levels=0),  # just past one CTA
    dict(B=1, n_q=3, q_pos0=4 * 40001 - 3, m=4, Nc=40001, k=1000, tie_levels=0),  # odd row pitch, ragged tail
    dict(B=1, n_q=2, q_pos0=4 * 524288 - 2, m=4, Nc=524288, k=2000, tie_levels=0),  # longest row
    dict(B=1, n_q=2, q_pos0=4 * 524288 - 2, m=4, Nc=524288, k=4096, tie_levels=0),  # streamed route only
])
def test_topk_bit_exact(case):
    _topk_case(seed=sum(case.values()) % 1000, **case)


@pytest.mark.parametrize("Nc", [5000, 20000, 262144])
def test_topk_infinite_scores(Nc):
    """Rows holding +inf and -inf scores, for each row-length route (staged
    keys, one fused CTA, chunked collection): infinities rank above and below
    every finite score, equal ones by index."""
    _topk_case(B=2, n_q=1, q_pos0=4 * Nc - 1, m=4, Nc=Nc, k=1024, tie_levels=0, seed=90, plant_inf=40)


@pytest.mark.parametrize("order", ["ascending", "descending"])
def test_topk_clustered_rows(order):
    """Rows whose best entries sit together (in the last or first chunk)."""
    _topk_case(B=2, n_q=1, q_pos0=(1 << 20) - 1, m=4, Nc=262144, k=1024, tie_levels=0, seed=77, order=order)
