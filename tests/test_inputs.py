"""The seeded generators: deterministic, per-sequence, and shaped as the
named workloads state."""
import torch

from long_context_compressed_18_b300 import configs, inputs


def test_deterministic_and_batch_independent():
    s = configs.shape(name="t", kind="csa", B=3, n=64, m=4, n_q=64, q_pos0=0, H=2, d=8,
                      H_I=2, d_I=32, k=4, idx_q_dtype="e4m3")
    a = inputs.make_inputs(s)
    b = inputs.make_inputs(s)
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key
    one = inputs.make_inputs(s, batches=[2])
    assert torch.equal(one["k"][0], a["k"][2])
    assert a["idx_q"].dtype == torch.uint8 and a["idx_q_scale"].shape == (3, 64, 2)


def test_decode_shapes():
    s = configs.shape(name="t", kind="csa_decode", B=2, n=4096, m=4, n_q=1, q_pos0=4095,
                      H=4, d=16, H_I=4, d_I=128, k=8, idx_q_dtype="e4m3", idx_k_dtype="e4m3")
    x = inputs.make_inputs(s)
    assert x["k_c"].shape == (2, 1024, 16) and x["k_c"].dtype == torch.bfloat16
    assert x["idx_k_c"].shape == (2, 1024, 128) and x["idx_k_c_scale"].shape == (2, 1024)
    # decoded row maximum equals amax: code 448 times scale amax/448
    v = x["idx_k_c"].view(torch.float8_e4m3fn).float().abs().amax(-1)
    assert torch.all(v == 448.0)


def test_random_index_sets_valid():
    s = configs.shape(name="t", kind="csa", B=1, n=64, m=4, n_q=64, q_pos0=0, H=1, d=8, k=5)
    idx = inputs.random_index_sets(s, seed=3)
    for i in range(64):
        nv = s.nv(i)
        row = idx[0, i]
        c = min(5, nv)
        assert torch.all(row[c:] == -1)
        sel = row[:c]
        assert torch.all(sel[1:] > sel[:-1]) and torch.all((sel >= 0) & (sel < nv))
