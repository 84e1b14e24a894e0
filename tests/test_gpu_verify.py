"""GPU parity of the speculative verify step (dspark_verify) against the fp64 oracle.

Rules (as for the draft sampler): accepted counts and tokens are bit-exact, except at a
near-tie, where fp32 and fp64 may legitimately decide differently:
  * an accept decision whose oracle margin |(ln q - ln p)(x_j) - ln a_j| is below 1e-4;
  * a correction / bonus draw whose oracle winner and runner-up scores differ by less than
    1e-4 (the GPU's token must then be the runner-up).
Near-ties are counted; a request is compared up to its first one.
"""
import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from oracle import oracle
from semi_autoregressive_drafting_gb300 import inputs

pytestmark = pytest.mark.gpu

TIE = 1e-4


def check(o, n, toks):
    """Compare GPU results with the oracle's; returns the number of near-ties."""
    ties = 0
    G = o.margin.shape[1]
    for b in range(len(n)):
        if o.n_accepted[b] < 0:
            assert n[b] == -1 and np.all(toks[b] == -1)
            continue
        m = o.margin[b]
        tested = int(min(o.n_accepted[b] + 1, G))
        if np.any(np.abs(m[:tested]) < TIE):  # a near-tie among the decisions
            ties += 1
            continue
        assert n[b] == o.n_accepted[b], (b, n[b], o.n_accepted[b], m)
        k = n[b]
        assert np.array_equal(toks[b, :k], o.tokens[b, :k]), b
        assert np.all(toks[b, k + 1:] == -1), b
        if toks[b, k] != o.tokens[b, k]:
            gap = o.best[b] - o.best2[b]
            assert toks[b, k] == o.tokens2[b] and gap < TIE, (b, toks[b, k], o.tokens[b, k], gap)
            ties += 1
    return ties


def run_case(B, G, V, *, seed, T=1.0, tokens="uniform", noise=1.0, vseed=7, identical=None):
    t = inputs.verify_inputs(B, G, V, seed=seed, target_noise=noise, tokens=tokens)
    if identical is not None:  # these requests' target rows equal their draft rows: accept all
        t["target_logits"][identical, :G] = t["draft_logits"][identical]
    o = oracle.verify(gamma=G, T=T, seed=vseed, draft_logits=t["draft_logits"].numpy(),
                      target_logits=t["target_logits"].numpy(),
                      draft_tokens=t["draft_tokens"].numpy())
    d = {k: v.cuda() for k, v in t.items()}
    ws = ds.VerifyWorkspace(B, G, V)
    n, toks = ds.verify(d["draft_logits"], d["target_logits"], d["draft_tokens"], T=T, seed=vseed,
                        workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == (1 if o.status else 0)
    ties = check(o, n.cpu().numpy(), toks.cpu().numpy())
    # a second call on the same workspace gives the same answer (it resets itself)
    n2, toks2 = ds.verify(d["draft_logits"], d["target_logits"], d["draft_tokens"], T=T,
                          seed=vseed, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(n, n2) and torch.equal(toks, toks2)
    print(f"verify B={B} gamma={G} V={V}: accepted mean {o.n_accepted.mean():.2f}, near-ties {ties}")
    return o, ties


@pytest.mark.parametrize("B,G,V,tokens", [(5, 3, 5000, "uniform"), (64, 7, 40000, "argmax"),
                                          (37, 16, 20001, "uniform"), (1, 1, 2, "uniform"),
                                          (128, 15, 8192, "argmax"),
                                          (130, 4, 16384 * 2 + 4, "argmax")])
def test_verify_matches_oracle(B, G, V, tokens):
    o, ties = run_case(B, G, V, seed=200 + B, tokens=tokens)
    assert ties <= max(1, B // 50)


def test_verify_temperature_and_accept_all():
    o, ties = run_case(24, 5, 12000, seed=310, T=0.7, tokens="argmax", identical=[0, 3, 7])
    assert np.all(o.n_accepted[[0, 3, 7]] == 5)  # p = q: the whole block and a bonus
    assert ties <= 1


def test_verify_rejects_everything_for_distant_target():
    # a target far from the draft: most first positions reject, the correction path dominates
    o, ties = run_case(48, 6, 9000, seed=320, noise=6.0)
    assert (o.n_accepted == 0).mean() > 0.5
    assert ties <= 1


def test_verify_invalid_token():
    B, G, V = 6, 3, 1000
    t = inputs.verify_inputs(B, G, V, seed=330)
    t["draft_tokens"][2, 1] = V
    d = {k: v.cuda() for k, v in t.items()}
    ws = ds.VerifyWorkspace(B, G, V)
    n, toks = ds.verify(d["draft_logits"], d["target_logits"], d["draft_tokens"], seed=1, workspace=ws)
    assert ws.status() == 1
    n = n.cpu().numpy()
    assert n[2] == -1 and np.all(toks[2].cpu().numpy() == -1)
    assert np.all(np.delete(n, 2) >= 0)


@pytest.mark.slow
def test_verify_qwen3_8b_shape():
    # the labelled workload's shape: B = 64, gamma = 7, V = 151936
    o, ties = run_case(64, 7, 151936, seed=340, tokens="argmax")
    assert ties <= 1
