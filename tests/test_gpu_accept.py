"""GPU parity of lbx_accept_walk (verify argmax + greedy acceptance walk)
against the oracle: bit-exact argmax, accepted node and next token."""
import numpy as np
import pytest
import torch

import oracle
from tree_verify_linear_gb300 import lbx
from tree_verify_linear_gb300.inputs import ACCEPT_VOCAB, make_accept_inputs

pytestmark = pytest.mark.gpu


def run_accept(inp, ws=None, logits_offset=0, with_argmax=True):
    Bq, N, V = inp["logits"].shape
    flat = np.zeros(Bq * N * V + logits_offset, dtype=np.float32)
    flat[logits_offset:] = inp["logits"].reshape(-1)
    lg_all = torch.from_numpy(flat).cuda()
    lg = lg_all[logits_offset:].view(Bq, N, V)
    dr = torch.from_numpy(inp["draft"]).cuda()
    pa = torch.from_numpy(inp["parent"]).cuda()
    acc = torch.full((Bq,), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((Bq,), -7, dtype=torch.int32, device="cuda")
    am = torch.full((Bq, N), -7, dtype=torch.int32, device="cuda") if with_argmax else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = lbx.new_accept_workspace(Bq, N, V) if ws is None else ws
    lbx.lbx_accept_walk(lg, dr, pa, acc, nxt, ws, argmax_out=am, d_status=st)
    torch.cuda.synchronize()
    return (None if am is None else am.cpu().numpy(), acc.cpu().numpy(), nxt.cpu().numpy(),
            int(st.item()), ws)


def check(inp, **kw):
    am, acc, nxt, st, ws = run_accept(inp, **kw)
    assert st == 0
    am_r, acc_r, nxt_r = oracle.accept_walk(inp["logits"], inp["draft"], inp["parent"])
    if am is not None:
        assert np.array_equal(am, am_r)
    assert np.array_equal(acc, acc_r)
    assert np.array_equal(nxt, nxt_r)
    return ws


def test_serving_batch_full_vocab():
    """5 requests, budget-22 DDTree-shaped trees, 152K vocabulary."""
    check(make_accept_inputs(5, 22, ACCEPT_VOCAB, seed=2001))


def test_ties_and_sibling_collisions():
    check(make_accept_inputs(5, 22, ACCEPT_VOCAB, seed=2002, ties=True))


@pytest.mark.parametrize("V", [1, 3, 7, 1001, 2048, 4097, 65537])
def test_ragged_vocab_and_misaligned_rows(V):
    inp = make_accept_inputs(2, 9, V, seed=2003 + V, tree="uniform")
    check(inp)
    check(inp, logits_offset=1)  # rows start off the 16-byte grid


def test_single_node_and_no_argmax_output():
    inp = make_accept_inputs(3, 1, 5000, seed=2010)
    check(inp, with_argmax=False)


def test_long_chain_full_match():
    """4096-token chain whose every token matches: the walk reaches the end."""
    N, V = 4096, 64
    rng = np.random.default_rng(2011)
    lg = rng.standard_normal((1, N, V), dtype=np.float32)
    pa = np.arange(-1, N - 1, dtype=np.int32)[None]
    dr = np.zeros((1, N), np.int32)
    dr[0, 1:] = np.argmax(lg[0, :-1], axis=-1)  # test-side planting only
    dr[0, 3000] = (dr[0, 3000] + 1) % V         # the match breaks at 3000
    check({"logits": lg, "draft": dr, "parent": pa})


def test_nan_inf_rows():
    inp = make_accept_inputs(2, 12, 3000, seed=2012, tree="uniform")
    lg = inp["logits"]
    lg[0, 0, :100] = np.nan
    lg[0, 1, :] = np.nan
    lg[0, 2, :] = -np.inf
    lg[0, 2, 17] = np.nan
    lg[1, 3, ::7] = np.inf
    check(inp)


def test_workspace_reuse_across_calls():
    """The arrival counters are cleared by each call: a second call on the
    same workspace (other inputs) is correct too."""
    ws = check(make_accept_inputs(4, 22, 20000, seed=2013))
    check(make_accept_inputs(4, 22, 20000, seed=2014), ws=ws)
    assert not ws.cpu().numpy()[-256:].any()


def test_invalid_tree_sets_status_and_writes_nothing():
    inp = make_accept_inputs(2, 6, 500, seed=2015)
    inp["parent"][1, 4] = 5  # parent not before the node
    am, acc, nxt, st, _ = run_accept(inp)
    assert st == lbx.LBX_ETREE
    assert acc[1] == -7 and nxt[1] == -7 and (am[1] == -7).all()
    # the valid request is still processed
    am_r, acc_r, nxt_r = oracle.accept_walk(inp["logits"][:1], inp["draft"][:1],
                                            inp["parent"][:1])
    assert acc[0] == acc_r[0] and nxt[0] == nxt_r[0] and np.array_equal(am[0], am_r[0])


def test_host_argument_checks():
    lg = torch.zeros((1, 2, 8), dtype=torch.float32, device="cuda")
    i1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    i2 = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    ws = lbx.new_accept_workspace(1, 2, 8)
    with pytest.raises(lbx.LbxError):
        lbx.lbx_accept_walk(lg, i2, i2, i1, i1, ws[:8])  # short workspace
    assert lbx.lbx_accept_workspace_size(1, lbx.LBX_ACCEPT_MAX_NODES + 1, 8) == 0
