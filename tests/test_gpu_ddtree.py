"""GPU parity of lbx_ddtree_build (best-first DDTree construction from the
draft's top-K scores) against the oracle: bit-exact parents, tokens, depths,
scores and node counts; and its tree fed to lbx_verify_step."""
import numpy as np
import pytest
import torch

import oracle
from tree_verify_linear_gb300 import lbx
from tree_verify_linear_gb300.inputs import ACCEPT_VOCAB, make_draft_topk

pytestmark = pytest.mark.gpu


def run_build(d, B, with_opt=True):
    Bq, D, K = d["logp"].shape
    lp = torch.from_numpy(np.ascontiguousarray(d["logp"])).cuda()
    tk = torch.from_numpy(np.ascontiguousarray(d["tok"])).cuda()
    rt = torch.from_numpy(d["root_tok"]).cuda()
    par = torch.full((Bq, B), -7, dtype=torch.int32, device="cuda")
    tn = torch.full((Bq, B), -7, dtype=torch.int32, device="cuda")
    dp = torch.full((Bq, B), -7, dtype=torch.int32, device="cuda") if with_opt else None
    sc = torch.full((Bq, B), 7.0, dtype=torch.float32, device="cuda") if with_opt else None
    nn = torch.full((Bq,), -7, dtype=torch.int32, device="cuda")
    lbx.lbx_ddtree_build(lp, tk, rt, B, par, tn, nn, depth_out=dp, score_out=sc)
    torch.cuda.synchronize()
    out = [par.cpu().numpy(), tn.cpu().numpy(), None if dp is None else dp.cpu().numpy(),
           None if sc is None else sc.cpu().numpy(), nn.cpu().numpy()]
    return out


def check(d, B, with_opt=True):
    par, tn, dp, sc, nn = run_build(d, B, with_opt)
    rp, rt, rd, rs, rn = oracle.ddtree_build(d["logp"], d["tok"], d["root_tok"], B)
    assert np.array_equal(nn, rn)
    assert np.array_equal(par, rp)
    assert np.array_equal(tn, rt)
    if with_opt:
        assert np.array_equal(dp, rd)
        assert np.array_equal(sc.view(np.int32), rs.view(np.int32))  # bit-exact
    return par, tn, nn


def test_budget22_draft_block16_top8():
    """Budget 22 from a 16-position draft block with top-8 tokens, 9 requests
    (more than one CTA of four warps)."""
    check(make_draft_topk(9, 16, 8, ACCEPT_VOCAB, seed=4001), 22)


@pytest.mark.parametrize("D,K,B", [(0, 3, 5), (1, 1, 4), (3, 2, 64), (6, 1, 22), (16, 8, 64),
                                   (64, 8, 64), (2, 8, 64), (5, 3, 1)])
def test_shapes(D, K, B):
    check(make_draft_topk(3, D, K, 5000, seed=4002 + 13 * D + K), B)


def test_ties_and_infinities():
    d = make_draft_topk(4, 6, 4, 1000, seed=4010)
    lp = d["logp"]
    lp[0] = np.log(np.float32(0.25))     # every score ties within a depth
    lp[1, :, 2:] = -np.inf               # unreachable tokens
    lp[2, 3] = lp[2, 3, ::-1].copy()     # a position not sorted
    check(d, 40)


def test_no_optional_outputs():
    check(make_draft_topk(5, 10, 4, 3000, seed=4011), 22, with_opt=False)


def test_tree_feeds_verify_step():
    """The built tree (budget 22) drives lbx_verify_step: same o and state as
    the oracle's verify on that tree."""
    from gpu_util import check_verify, run_verify
    from tree_verify_linear_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["layer27b"]
    inp = make_inputs(w)
    d = make_draft_topk(w.Bq, 16, 8, ACCEPT_VOCAB, seed=4012)
    par, _, nn = check(d, w.N)
    assert (nn == w.N).all()
    inp["parent"] = np.ascontiguousarray(par.reshape(w.Bq, w.N))
    inp["accepted"][:] = np.int32(w.N - 1)
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == 0
    check_verify(w, inp, o, st, cc)


def test_host_argument_checks():
    lp = torch.zeros((1, 2, 9), dtype=torch.float32, device="cuda")  # K = 9 > 8
    tk = torch.zeros((1, 2, 9), dtype=torch.int32, device="cuda")
    rt = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(lbx.LbxError):
        lbx.lbx_ddtree_build(lp, tk, rt, 4, o, o, n)
    with pytest.raises(lbx.LbxError):
        lbx.lbx_ddtree_build(lp[:, :, :8].contiguous(), tk[:, :, :8].contiguous(), rt, 65,
                             torch.zeros((1, 65), dtype=torch.int32, device="cuda"),
                             torch.zeros((1, 65), dtype=torch.int32, device="cuda"), n)
