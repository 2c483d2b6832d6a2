"""Context-parallel CSA decode of one sequence on CPU ranks (gloo): the
entry-range shards, local indexer + top-k, the all-gather of (score, index)
candidates, the global select, partial attention with lse and the rank-order
combine must reproduce the unsharded oracle -- the selection bit for bit, the
output and lse within 1e-12."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

CASES = {
    # every entry visible, k well below the shard sizes
    "full": dict(Nc=3001, t=4 * 3001 - 1, k=256),
    # the query sees only part of the cache: the last shard is partly, or not at all, visible
    "partial": dict(Nc=3001, t=4 * 1700 + 2, k=256),
    # fewer visible entries than k: everything selected, -1 padded
    "short": dict(Nc=500, t=4 * 200 + 1, k=256),
}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(Nc, seed=3):
    from long_context_compressed_18_b300 import configs, inputs
    s = configs.shape(name="cp", kind="csa_decode", B=1, n=4 * Nc, m=4, n_q=1, q_pos0=4 * Nc - 1, H=8, d=64,
                      H_I=64, d_I=128, k=256, idx_q_dtype="e4m3", idx_k_dtype="e4m3", seed=seed)
    return inputs.make_inputs(s)


def _rank_main(rank, world, port, case, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import cp
        c = CASES[case]
        x = _inputs(c["Nc"])
        lo, hi = cp.shard_bounds(c["Nc"], rank, world)
        sel, out, lse = cp.cp_csa_decode(x["q"], x["idx_q"], x["idx_q_scale"], "e4m3", x["k_c"][:, lo:hi],
                                         x["v_c"][:, lo:hi], x["idx_k_c"][:, lo:hi], x["idx_k_c_scale"][:, lo:hi],
                                         "e4m3", c["t"], 4, c["k"], 1.0 / 8.0)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), sel=sel, out=out, lse=lse)
    finally:
        tdist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("case", sorted(CASES))
def test_cp_decode_matches_unsharded_oracle(tmp_path, world, case):
    import oracle
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, case, str(tmp_path)), nprocs=world, start_method="spawn")
    c = CASES[case]
    x = _inputs(c["Nc"])
    _, _, sel = oracle.csa_index_topk(x["idx_q"], x["idx_q_scale"], "e4m3", x["idx_k_c"], x["idx_k_c_scale"],
                                      "e4m3", c["t"], 4, c["k"])
    want_o, want_l = oracle.attention(x["q"], x["k_c"], x["v_c"], 1.0 / 8.0, oracle.SPARSE, idx=sel[None])
    nv = int(oracle.visible(c["t"], 4, c["Nc"]))
    assert (sel[0] >= 0).sum() == min(nv, c["k"])
    for r in range(world):
        got = np.load(tmp_path / f"rank{r}.npz")
        assert np.array_equal(got["sel"], sel[0].astype(np.int64)), r      # bit-identical selection
        assert np.max(np.abs(got["out"] - want_o[0])) <= 1e-12, r
        assert np.max(np.abs(got["lse"] - want_l[0])) <= 1e-12, r


def test_shard_bounds_cover_every_entry_once():
    from oracle import cp
    for n in (1, 7, 3001, 262144):
        for w in (1, 2, 3, 8):
            b = [cp.shard_bounds(n, r, w) for r in range(w)]
            assert b[0][0] == 0 and b[-1][1] == n
            assert all(b[i][1] == b[i + 1][0] for i in range(w - 1))
            assert max(h - l for l, h in b) - min(h - l for l, h in b) <= 1
