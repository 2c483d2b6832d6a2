"""GPU parity of the streaming decode state ("DeepSeek V4 技术解读" §2.1, KV
Cache 压缩, applied one generated token at a time):

* csa_decode_append, token by token from sequences of different starting
  lengths, fills exactly the cache entries whose blocks close, each equal to
  the oracle's compression of the whole stream (fp32 / bf16 / E4M3 / E2M1
  caches, m = 4 and m' = 128); entries that do not close are left untouched,
  the open block sits in the staging buffer bit for bit, and the device
  token counts advance by one a call.
* csa_index_topk_varlen selects, for each sequence's queries at their own
  positions lens[b] - n_q + i, the oracle's top-k (near-ties only), pads
  short sequences with -1, and equals csa_index_topk when all lengths agree.
* A block closing past the caches' capacity is not written and is reported
  through the device status word.
* A short streaming decode loop (append, select, attend) matches the oracle
  stage by stage."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import inputs, lib, pipeline
from helpers import (DEV, assert_close, check_attn_stagewise, check_e2m1_keys, host, sync_status,
                     topk_near_tie_check)

pytestmark = pytest.mark.gpu

_TORCH = {lib.F32: torch.float32, lib.BF16: torch.bfloat16}


def _arith_bound(lg, x, m, want, bf16_out):
    """fp32 token-order sums of m weighted terms, each weight within a few
    ulp: (m + 4) 2^-24 sum_i w_i |x_i| (the same compression over |x|), plus
    the bf16 rounding of the output where the cache is bf16."""
    mag = oracle.compress(lg, np.abs(np.asarray(x, np.float32)), m)
    b = (m + 4) * 2.0 ** -24 * mag * 1.01 + 1e-9
    if bf16_out:
        b = b + 2.0 ** -8 * np.abs(want)
    return b


@pytest.mark.parametrize("m,x_code,kv_code,ik_code", [
    (4, lib.BF16, lib.BF16, lib.E4M3),
    (4, lib.F32, lib.F32, lib.F32),
    (4, lib.BF16, lib.BF16, lib.E2M1),
    (128, lib.BF16, lib.BF16, lib.BF16),
    (128, lib.F32, lib.F32, lib.E4M3),
])
def test_decode_append_matches_compression(m, x_code, kv_code, ik_code):
    g = torch.Generator().manual_seed(m * 10 + ik_code)
    B, d, dI = 4, 128 if m == 4 else 64, 128
    L0 = [0, m + 1, 3 * m - 1, 1]                    # a ragged open block in three of four
    T = 2 * m + 3
    n_tot = [l + T for l in L0]
    nmax = max(n_tot)
    N_cap = nmax // m + 1
    xdt = _TORCH[x_code]
    lg = torch.randn(B, nmax, generator=g) * 2
    K = torch.randn(B, nmax, d, generator=g).to(xdt)
    V = torch.randn(B, nmax, d, generator=g).to(xdt)
    IK = torch.randn(B, nmax, dI, generator=g).to(xdt)

    # the state after L0[b] tokens: counts, and the open block in the staging buffer
    st_lg = torch.zeros(B, m)
    st_k, st_v, st_ik = torch.zeros(B, m, d, dtype=xdt), torch.zeros(B, m, d, dtype=xdt), torch.zeros(B, m, dI, dtype=xdt)
    for b, l in enumerate(L0):
        o = l - l % m
        st_lg[b, :l % m], st_k[b, :l % m], st_v[b, :l % m], st_ik[b, :l % m] = lg[b, o:l], K[b, o:l], V[b, o:l], IK[b, o:l]
    st_lg, st_k, st_v, st_ik = st_lg.to(DEV), st_k.to(DEV), st_v.to(DEV), st_ik.to(DEV)
    lens = torch.tensor(L0, dtype=torch.int64, device=DEV)

    kvdt = _TORCH[kv_code]
    k_c = torch.full((B, N_cap, d), float("nan"), dtype=kvdt, device=DEV)
    v_c = torch.full((B, N_cap, d), float("nan"), dtype=kvdt, device=DEV)
    if ik_code == lib.E4M3:
        ik_c = torch.full((B, N_cap, dI), 0xAB, dtype=torch.uint8, device=DEV)
        ik_s = torch.full((B, N_cap), float("nan"), device=DEV)
    elif ik_code == lib.E2M1:
        ik_c = torch.full((B, N_cap, dI // 2), 0xAB, dtype=torch.uint8, device=DEV)
        ik_s = torch.full((B, N_cap, dI // 32), 0xAB, dtype=torch.uint8, device=DEV)
    else:
        ik_c = torch.full((B, N_cap, dI), float("nan"), dtype=_TORCH[ik_code], device=DEV)
        ik_s = None

    # each step's new tokens: token L0[b] + t of sequence b
    pos = torch.tensor([[l + t for l in L0] for t in range(T)])
    ar = torch.arange(B)
    new_lg = torch.stack([lg[ar, pos[t]] for t in range(T)]).to(DEV)          # [T, B]
    new_k = torch.stack([K[ar, pos[t]] for t in range(T)]).to(DEV)
    new_v = torch.stack([V[ar, pos[t]] for t in range(T)]).to(DEV)
    new_ik = torch.stack([IK[ar, pos[t]] for t in range(T)]).to(DEV)
    for t in range(T):
        lib.csa_decode_append(B, m, d, dI, N_cap, new_lg[t], new_k[t], new_v[t], new_ik[t], x_code, st_lg, st_k,
                              st_v, st_ik, lens, k_c, v_c, kv_code, ik_c, ik_code, ik_s)
    sync_status()

    assert host(lens).tolist() == n_tot
    kch, vch, ikh = host(k_c).float().numpy(), host(v_c).float().numpy(), host(ik_c)
    iksh = None if ik_s is None else host(ik_s)
    for b in range(B):
        n = n_tot[b]
        j0, j1 = L0[b] // m, n // m                  # the entries closed by the appends
        assert j1 > j0
        for name, X, got in (("K", K, kch), ("V", V, vch)):
            want = oracle.compress(lg[b:b + 1, :n], X[b:b + 1, :n].float(), m)[0]
            bound = _arith_bound(lg[b:b + 1, :n], X[b:b + 1, :n].float(), m, want, kv_code == lib.BF16)[0]
            err = np.abs(got[b, j0:j1] - want[j0:j1])
            assert np.all(err <= bound[j0:j1]), (name, b, float(np.max(err - bound[j0:j1])))
            assert np.isnan(got[b, :j0]).all() and np.isnan(got[b, j1:]).all(), (name, b, "untouched entries")
        ref_full = oracle.compress(lg[b:b + 1, :n], IK[b:b + 1, :n].float(), m)
        ref = ref_full[0][j0:j1]
        if ik_code in (lib.F32, lib.BF16):
            gi = ikh[b].float().numpy()
            bound = _arith_bound(lg[b:b + 1, :n], IK[b:b + 1, :n].float(), m, ref_full,
                                 ik_code == lib.BF16)[0][j0:j1]
            assert np.all(np.abs(gi[j0:j1] - ref) <= bound)
            assert np.isnan(gi[:j0]).all() and np.isnan(gi[j1:]).all()
        elif ik_code == lib.E4M3:
            wc, ws = oracle.quant_e4m3_rows(ref.astype(np.float32))
            c, s = ikh[b, j0:j1].numpy(), iksh[b, j0:j1].numpy()
            assert_close(s, ws, atol=0, rtol=1e-6, what="e4m3 scales")
            dec = oracle.e4m3_decode(c).astype(np.float64) * s[..., None]
            want = oracle.e4m3_decode(wc).astype(np.float64) * ws[..., None]
            assert np.all(np.abs(dec - want) <= (np.abs(want) * 2.0 ** -3 + s[..., None] * 2.0 ** -9) * 1.0001)
            assert (ikh[b, :j0] == 0xAB).all() and (ikh[b, j1:] == 0xAB).all()
            assert torch.isnan(iksh[b, :j0]).all() and torch.isnan(iksh[b, j1:]).all()
        else:
            check_e2m1_keys(ikh[b, j0:j1].numpy(), iksh[b, j0:j1].numpy(), ref)
            assert (ikh[b, :j0] == 0xAB).all() and (ikh[b, j1:] == 0xAB).all()
        # the open block, bit for bit
        r, o = n % m, n - n % m
        assert torch.equal(host(st_lg)[b, :r], lg[b, o:n])
        for st, X in ((st_k, K), (st_v, V), (st_ik, IK)):
            assert torch.equal(host(st)[b, :r], X[b, o:n])


def test_decode_append_past_capacity_flags_and_writes_nothing():
    B, m, d, dI, N_cap = 2, 4, 64, 64, 2
    g = torch.Generator().manual_seed(3)
    state = pipeline.DecodeState(B, m, d, dI, N_cap, x_dtype=torch.float32, kv_dtype=torch.float32, ik_kind="f32")
    state.k_c.fill_(7.0)
    torch.cuda.synchronize()
    lib.csa_device_status()                          # start from a clear word
    for t in range(N_cap * m):                       # fills the caches exactly
        state.append(torch.randn(B, generator=g).to(DEV), torch.randn(B, d, generator=g).to(DEV),
                     torch.randn(B, d, generator=g).to(DEV), torch.randn(B, dI, generator=g).to(DEV))
    sync_status()                                    # no flag yet
    before = host(state.k_c).clone()
    for t in range(m):                               # the third block has no entry
        state.append(torch.randn(B, generator=g).to(DEV), torch.randn(B, d, generator=g).to(DEV),
                     torch.randn(B, d, generator=g).to(DEV), torch.randn(B, dI, generator=g).to(DEV))
    torch.cuda.synchronize()
    with pytest.raises(lib.CsaError) as e:
        lib.csa_device_status()
    assert e.value.status == 7                       # CSA_ERR_DEVICE
    assert torch.equal(host(state.k_c), before)
    assert host(state.lens).tolist() == [(N_cap + 1) * m] * B
    lib.csa_device_status()                          # read-and-clear


def test_decode_append_rejects_bad_arguments_on_the_host():
    t = torch.zeros(64, device=DEV)
    lens = torch.zeros(4, dtype=torch.int64, device=DEV)
    args = [t, t, t, t, lib.F32, t, t, t, t, lens, t, t, lib.F32, t, lib.F32]
    with pytest.raises(lib.CsaError) as e:
        lib.csa_decode_append(1, 129, 8, 8, 1, *args)            # m above 128
    assert e.value.status == 2
    with pytest.raises(lib.CsaError) as e:
        lib.csa_decode_append(1, 4, 8, 48, 1, *args[:-1], lib.E2M1, t)  # E2M1 needs d_I % 32 == 0
    assert e.value.status == 2
    with pytest.raises(lib.CsaError) as e:
        lib.csa_decode_append(1, 4, 8, 8, 1, *args[:-1], lib.E4M3, None)  # E4M3 without its scales
    assert e.value.status == 1


# ---- selection at per-sequence positions ------------------------------------------

def _idx_inputs(B, n_q, Nc, seed):
    g = torch.Generator().manual_seed(seed)
    q, qs = inputs.quantise_e4m3_lastdim(torch.randn(B, n_q, 64, 128, generator=g))
    k, ks = inputs.quantise_e4m3_lastdim(torch.randn(B, Nc, 128, generator=g))
    return q, qs, k, ks


@pytest.mark.parametrize("n_q", [1, 2])
@pytest.mark.parametrize("score", ["f32", "bf16"])
def test_index_topk_varlen_against_oracle(n_q, score):
    N_cap, k, m = 70000, 1024, 4
    lens = [4 * N_cap + 3, 4 * 5000 + 2, 4 * 40000 + 1, 4 * 500, n_q]   # the last sees no entry
    B = len(lens)
    q, qs, kk, ks = _idx_inputs(B, n_q, N_cap, seed=n_q * 7 + len(score))
    topk = torch.empty(B, n_q, k, dtype=torch.int32, device=DEV)
    sd = lib.F32 if score == "f32" else lib.BF16
    wb = lib.csa_index_topk_workspace_size(B, n_q, N_cap, 64, 128, k, lib.E4M3, sd)
    ws = lib.empty_workspace(wb)
    lib.csa_index_topk_varlen(B, n_q, torch.tensor(lens, dtype=torch.int64, device=DEV), m, N_cap, 64, 128, k,
                              q.to(DEV), lib.E4M3, qs.to(DEV), kk.to(DEV), lib.E4M3, ks.to(DEV), topk, ws, wb,
                              score_dtype=sd)
    sync_status()
    got = host(topk).numpy()
    for b, L in enumerate(lens):
        p0 = L - n_q
        s64, s32, sel = oracle.csa_index_topk(q[b:b + 1], qs[b:b + 1], "e4m3", kk[b:b + 1], ks[b:b + 1], "e4m3",
                                              p0, m, k)
        vis = oracle.visible(p0 + np.arange(n_q), m, N_cap)
        if score == "f32":
            topk_near_tie_check(got[b], sel, s64, vis, k)
        else:
            # bf16 storage: the selection is the exact top-k of the rounded
            # fp32 scores, so it holds only entries whose fp32 score is within
            # a bf16 step of the oracle's k-th
            for i in range(n_q):
                c = min(k, int(vis[i]))
                assert (got[b, i, c:] == -1).all()
                gs = got[b, i, :c]
                assert len(set(gs.tolist())) == c and (gs >= 0).all() and (gs < vis[i]).all()
                if c:
                    row = s64[i, :vis[i]]
                    sk = np.sort(row)[::-1][c - 1]
                    assert (s64[i, gs] >= sk - 2.0 ** -7 * abs(sk) - 1e-6 * np.abs(row).max()).all()


def test_index_topk_varlen_equals_uniform_route():
    B, n_q, N_cap, k = 3, 1, 60000, 512
    L = 4 * N_cap - 5
    q, qs, kk, ks = _idx_inputs(B, n_q, N_cap, seed=5)
    q, qs, kk, ks = q.to(DEV), qs.to(DEV), kk.to(DEV), ks.to(DEV)
    wb = lib.csa_index_topk_workspace_size(B, n_q, N_cap, 64, 128, k, lib.E4M3)
    ws = lib.empty_workspace(wb)
    a = torch.empty(B, n_q, k, dtype=torch.int32, device=DEV)
    b = torch.empty_like(a)
    lib.csa_index_topk(B, n_q, L - n_q, 4, N_cap, 64, 128, k, q, lib.E4M3, qs, kk, lib.E4M3, ks, a, ws, wb)
    lib.csa_index_topk_varlen(B, n_q, torch.full((B,), L, dtype=torch.int64, device=DEV), 4, N_cap, 64, 128, k, q,
                              lib.E4M3, qs, kk, lib.E4M3, ks, b, ws, wb)
    sync_status()
    assert torch.equal(a, b)


# ---- a short streaming decode loop ----------------------------------------------------

@pytest.mark.parametrize("ik_kind", ["e4m3", "e2m1"])
def test_streaming_decode_loop_stagewise(ik_kind):
    """Sequences of different lengths grow token by token; after each
    append every sequence's new query selects among its closed entries and
    attends to them.  Each stage is checked against the oracle on the same
    inputs: the caches against the oracle's compression, the selection
    against the oracle's top-k of the GPU-written keys (near-ties only), the
    attention against the oracle on the GPU's selection."""
    B, m, d, dI, H, k = 3, 4, 128, 128, 64, 64
    L0 = [4 * 300 + 1, 4 * 40, 4 * 17 + 3]
    T = 6
    nmax = max(L0) + T
    N_cap = nmax // m + 1
    g = torch.Generator().manual_seed(21)
    lg = torch.randn(B, nmax, generator=g) * 2
    K = (torch.randn(B, nmax, d, generator=g) * d ** -0.25).to(torch.bfloat16)
    V = torch.randn(B, nmax, d, generator=g).to(torch.bfloat16)
    IK = torch.randn(B, nmax, dI, generator=g).to(torch.bfloat16)
    st = pipeline.DecodeState(B, m, d, dI, N_cap, ik_kind=ik_kind)
    # the prefix: its closed blocks through the compression kernel, the open block staged
    for b, l in enumerate(L0):
        nc = l // m
        (kc, _), (vc, _), (ikc, iks) = pipeline.compress(lg[b:b + 1, :nc * m].to(DEV),
                                                         [K[b:b + 1, :nc * m].to(DEV), V[b:b + 1, :nc * m].to(DEV),
                                                          IK[b:b + 1, :nc * m].to(DEV)], m, ["bf16", "bf16", ik_kind])
        st.k_c[b, :nc], st.v_c[b, :nc], st.ik_c[b, :nc], st.ik_scale[b, :nc] = kc[0], vc[0], ikc[0], iks[0]
        o = nc * m
        st.stage_logits[b, :l - o] = lg[b, o:l].to(DEV)
        st.stage_k[b, :l - o], st.stage_v[b, :l - o], st.stage_ik[b, :l - o] = (K[b, o:l].to(DEV), V[b, o:l].to(DEV),
                                                                                  IK[b, o:l].to(DEV))
    st.lens.copy_(torch.tensor(L0))
    ws = pipeline.Workspace()
    ar = torch.arange(B)
    tau = 1 / math.sqrt(d)
    for t in range(T):
        p = torch.tensor(L0) + t
        st.append(lg[ar, p].contiguous().to(DEV), K[ar, p].contiguous().to(DEV), V[ar, p].contiguous().to(DEV),
                  IK[ar, p].contiguous().to(DEV))
        q_idx, q_s = inputs.quantise_e4m3_lastdim(torch.randn(B, 1, 64, dI, generator=g))
        q = (torch.randn(B, 1, H, d, generator=g) * d ** -0.25).to(torch.bfloat16)
        topk = st.select(q_idx.to(DEV), "e4m3", q_s.to(DEV), k, ws)
        out, lse = st.attend(q.to(DEV), topk, tau, ws)
        sync_status()
        n = p + 1
        assert host(st.lens).tolist() == n.tolist()
        ikc, iks = host(st.ik_c), host(st.ik_scale)
        sel = host(topk).numpy()
        for b in range(B):
            nb = int(n[b])
            # stage 1: the caches' entries against the oracle's compression
            want_k = oracle.compress(lg[b:b + 1, :nb], K[b:b + 1, :nb].float(), m)[0]
            gk = host(st.k_c[b, :nb // m]).float().numpy()
            assert np.all(np.abs(gk - want_k) <= 2.0 ** -8 * np.abs(want_k) + 1e-5), b
            # stage 2: selection over the GPU-written keys
            s64, _, want_sel = oracle.csa_index_topk(q_idx[b:b + 1], q_s[b:b + 1], "e4m3", ikc[b:b + 1],
                                                     iks[b:b + 1], ik_kind, nb - 1, m, k)
            topk_near_tie_check(sel[b], want_sel, s64, [min(nb // m, N_cap)], k)
        # stage 3: attention on the GPU's selection over the GPU-written caches
        kc_h, vc_h = host(st.k_c).float(), host(st.v_c).float()
        want_o, want_l = oracle.attention(q.float(), kc_h, vc_h, tau, oracle.SPARSE, idx=sel)
        mag, _ = oracle.attention(q.float(), kc_h, vc_h.abs(), tau, oracle.SPARSE, idx=sel)
        check_attn_stagewise(host(out).float().numpy(), host(lse).numpy(), want_o, want_l, mag, f"step {t}")
