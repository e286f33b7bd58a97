"""Beam selection (xGR section 2.2, xBeam early sort termination) through the C ABI, against
the oracle's full sort on the same seeded candidate lists: parents, tokens and scores must
match bit for bit (the selection is unique: equal scores go to the smaller flat index)."""

import numpy as np
import pytest
import torch

import oracle
from decode_attention_xattention_gb300 import workloads as wl
from decode_attention_xattention_gb300 import xattn


def run_select(bs, lp, tok, W):
    R, BW, K = lp.shape
    dev = "cuda"
    d_bs, d_lp, d_tok = (torch.from_numpy(a).to(dev) for a in (bs, lp, tok))
    par = torch.full((R, W), -7, dtype=torch.int32, device=dev)
    tk = torch.full((R, W), -7, dtype=torch.int32, device=dev)
    sc = torch.full((R, W), float("nan"), dtype=torch.float32, device=dev)
    xattn.check(xattn.xattn_beam_select(R, BW, K, W, d_bs, d_lp, d_tok, par, tk, sc))
    torch.cuda.synchronize()
    return par.cpu().numpy(), tk.cpu().numpy(), sc.cpu().numpy()


def check_against_oracle(bs, lp, tok, W):
    want = oracle.load().beam_select(bs, lp, tok, W)
    got = run_select(bs, lp, tok, W)
    for name, g, w in zip(("parent", "token", "score"), got, want):
        np.testing.assert_array_equal(g, w, err_msg=name)
    return got


@pytest.mark.gpu
def test_hand_example():
    bs = np.array([[-1.0, -0.5, -3.0]], np.float32)
    lp = np.array([[[-0.25, -0.75, -2.0], [-0.75, -1.0, -1.5], [0.0, -0.125, -0.25]]], np.float32)
    tok = np.array([[[1, 2, 3], [11, 12, 13], [21, 22, 23]]], np.int32)
    par, tk, sc = check_against_oracle(bs, lp, tok, 6)
    assert par.tolist() == [[0, 1, 1, 0, 1, 0]] and tk.tolist() == [[1, 11, 12, 2, 13, 3]]


@pytest.mark.gpu
@pytest.mark.parametrize("R,BW,K,W", [(8, 128, 128, 128), (4, 512, 512, 512), (2, 7, 5, 20), (3, 100, 3, 1),
                                      (2, 4, 50, 200), (1, 1024, 1, 1024), (2, 16, 64, 1000), (5, 33, 17, 64)],
                         ids=["gr_128x128", "wide_512x512", "odd", "W1", "W_gt_BW_and_K", "all_candidates",
                              "W1000", "ragged"])
def test_shapes(R, BW, K, W):
    bs, lp, tok = wl.make_candidates(R, BW, K, seed=R * 1000 + BW + K + W)
    check_against_oracle(bs, lp, tok, W)


@pytest.mark.gpu
@pytest.mark.parametrize("R,BW,K,W,levels", [(4, 128, 128, 128, 3), (2, 64, 32, 300, 2), (3, 9, 7, 40, 5),
                                             (1, 512, 64, 512, 4)])
def test_many_equal_scores(R, BW, K, W, levels):
    """Few distinct values: long runs of equal scores, across beams and within one list,
    decided by the flat index, also at the cut."""
    bs, lp, tok = wl.make_candidates(R, BW, K, seed=levels + W, tie_levels=levels)
    check_against_oracle(bs, lp, tok, W)


@pytest.mark.gpu
def test_masked_candidates_and_signed_zero():
    """-inf (masked) tails, and scores of both signs of zero, which rank as equal."""
    bs, lp, tok = wl.make_candidates(3, 40, 20, seed=5, masked_frac=0.6)
    check_against_oracle(bs, lp, tok, 600)  # more than the unmasked candidates: -inf ones fill the tail
    bs = np.zeros((1, 4), np.float32)
    bs[0, 1] = -0.0
    lp = np.zeros((1, 4, 2), np.float32)
    lp[0, :, 1] = -1.0
    lp[0, 2, 0] = -0.0
    tok = np.arange(8, dtype=np.int32).reshape(1, 4, 2)
    par, _, _ = check_against_oracle(bs, lp, tok, 5)
    assert par.tolist() == [[0, 1, 2, 3, 0]]


@pytest.mark.gpu
def test_early_termination_leaves_lists_unread():
    """Beams that cannot enter the best W stop after a few positions: half the beams score
    -1e6 lower; at list position 0 they fill the empty array, at position 1 the other beams'
    candidates push them out, and by position 2 each of them meets a full array it cannot
    enter. Their
    lists past position 2 are poisoned with NaN, which would win every comparison it entered
    (and which the oracle's full scan rejects): the selection must come out unchanged."""
    R, BW, K, W = 2, 64, 64, 64
    bs, lp, tok = wl.make_candidates(R, BW, K, seed=21)
    low = np.arange(BW) >= BW // 2
    bs[:, low] = -1e6
    want = oracle.load().beam_select(bs, lp, tok, W)
    assert not np.isin(want[0], np.nonzero(low)[0]).any()
    lp_p = lp.copy()
    lp_p[:, low, 3:] = np.nan
    got = run_select(bs, lp_p, tok, W)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)
