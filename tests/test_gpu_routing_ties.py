"""Exact ties in the biased top-k, on the GPU through the C ABI
(lmoe_route_static, which takes the scores and the bias directly), against
the oracle's top-k and stable grouping.  The selection compares
u = fp32(s + b); among equal u the lower expert id wins, and the chosen ids
are listed by descending u, then ascending id (a reading: the pages do not
say how ties break).  Random scores almost never tie, so the ties are planted:
duplicated score columns, rows of all-equal scores, biases that make two
experts' u equal, bias steps too small to survive the fp32 add, a tie across
the k-th place, and a tie of 40 experts at the top (more candidates than the
selection's one-sort path takes)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_moe_layer_bias_gb300 as m
    m.load_library()
    return m


def planted(T, E, seed):
    rng = np.random.default_rng(seed)
    s = rng.random((T, E)).astype(np.float32)
    b = ((rng.random(E) - 0.5) * 0.05).astype(np.float32)
    for j in range(0, E - 1, 7):              # duplicated columns on every third row
        s[::3, j + 1] = s[::3, j]
        b[j + 1] = b[j]
    s[1, :] = 0.5                              # rows of all-equal scores
    s[T // 2, :] = 0.25
    # equal u through the bias (exact in fp32), on the last two experts:
    # 0.75 + 0 == 0.5 + 0.25
    b[E - 2], b[E - 1] = np.float32(0.0), np.float32(0.25)
    s[2, E - 2], s[2, E - 1] = np.float32(0.75), np.float32(0.5)
    # a bias step below half an ulp of s is absorbed by the fp32 add:
    # 0.5 + 2^-26 == 0.5 (the two experts before them)
    b[E - 4], b[E - 3] = np.float32(0.0), np.float32(2.0 ** -26)
    s[4, E - 4], s[4, E - 3] = np.float32(0.5), np.float32(0.5)
    return s, b


def with_boundary_tie(s, b, k):
    """Row 3: experts 0 .. k+3 tie at u = 0.9 above every other expert."""
    E = s.shape[1]
    n = min(E, k + 4)
    b[:n] = 0.0
    s[3, :] = (s[3, :] * 0.2).astype(np.float32)
    s[3, :n] = 0.9
    return s, b


def with_wide_tie(s, b):
    """Row 5: experts 8 .. 47 tie at u = 0.99 above every other expert.  Each
    of the 32 lanes then holds a key equal to the k-th largest, so more than
    32 keys reach the selection's threshold and the token takes the
    round-by-round path; the lowest ids win.  (E >= 48 only: with E <= 32
    every lane holds one key and the threshold never admits more than 32.)"""
    E = s.shape[1]
    if E >= 48:
        b[8:48] = 0.0
        s[5, :] = (s[5, :] * 0.2).astype(np.float32)
        s[5, 8:48] = 0.99
    return s, b


@pytest.mark.parametrize("T,E,k,seed", [(300, 896, 16, 1), (257, 64, 8, 2), (40, 12, 5, 3)])
def test_route_static_ties_match_the_oracle(lm, T, E, k, seed):
    s, b = with_wide_tie(*with_boundary_tie(*planted(T, E, seed), k))
    cfg = oracle.LayerConfig(d=64, latent=128, n_experts=E, top_k=k, inter=64, n_shared=1, shared_inter=64)
    u = (s + b[None, :]).astype(np.float32)
    assert any(len(set(row.tolist())) < E for row in u)      # the planting made ties
    idx_ref, gate_ref, _ = oracle.topk(cfg, s, b)
    counts, offsets, perm, inv = oracle.permute(cfg, idx_ref)

    got = lm.lmoe_route_static(torch.from_numpy(s).cuda(), torch.from_numpy(b).cuda(), k)
    torch.cuda.synchronize()
    idx = got["topk_idx"].cpu().numpy()
    assert np.array_equal(idx, idx_ref)
    assert np.array_equal(idx[3], np.arange(k))          # the boundary tie: lower ids win
    if E >= 48:
        assert np.array_equal(idx[5], np.arange(8, 8 + k))   # the wide tie
    assert np.array_equal(got["gates"].cpu().numpy().view(np.uint32), gate_ref.view(np.uint32))
    for key, ref in (("counts", counts), ("offsets", offsets), ("perm", perm), ("inv", inv)):
        assert np.array_equal(got[key].cpu().numpy(), ref), key
    # the order within a token: descending u, equal u by ascending id
    for t in range(T):
        uu = u[t, idx[t]]
        assert all(uu[j] > uu[j + 1] or (uu[j] == uu[j + 1] and idx[t, j] < idx[t, j + 1])
                   for j in range(k - 1)), t
