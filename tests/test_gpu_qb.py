"""GPU parity of the Quantile Balancing histogram (bit-exact counts) and the
quantile/bias read, through the C ABI, against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_bias_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_moe_layer_bias_gb300 as m
    m.load_library()
    return m


def hist_np(h: torch.Tensor) -> np.ndarray:
    return h.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("T,E,B", [(65536, 896, 1000), (4096, 128, 1000), (4099, 896, 10000),
                                   (1000, 40, 37), (1, 896, 1000),
                                   (3000, 24, 60000),    # bins beyond shared memory: global counters
                                   (200000, 64, 10000),  # 16-bit counters, several token chunks
                                   (70001, 32, 9999),    # 16-bit counters, odd B (last word half used)
                                   (5000, 1, 1000)])     # a single expert (scalar path)
def test_histogram_bit_exact(lm, T, E, B):
    s = synth.qb_scores(T, E, seed=T + E + B)
    s[0, 0] = 1.0
    s[-1, -1] = 0.0
    hg = lm.qb_histogram(s.cuda(), B)
    torch.cuda.synchronize()
    ref = oracle.qb_histogram(s.numpy(), B)
    assert np.array_equal(hist_np(hg), ref)
    assert hist_np(hg).sum(dtype=np.uint64) == T * E


def test_histogram_16bit_counters_do_not_carry(lm):
    """Large B packs two 16-bit counters per word; one bin receiving every
    token (T > 65535) must not carry into its neighbour: a counter that has
    reached 32768 after a span of 32768 rows goes to the global histogram."""
    T, E, B = 140000, 32, 10000
    s = synth.qb_scores(T, E, seed=5)
    s[:, 0] = 0.5          # bin 5000: an even bin, the low half of its word
    s[:, 1] = 0.50005      # bin 5000 as well (0.50005 * 10000 = 5000.5)
    s[:, 2] = 0.5001       # bin 5001: the high half of the same word
    hg = lm.qb_histogram(s.cuda(), B)
    torch.cuda.synchronize()
    h = hist_np(hg)
    assert h[0, 5000] == T and h[1, 5000] == T and h[2, 5001] == T
    assert np.array_equal(h, oracle.qb_histogram(s.numpy(), B))


def test_histogram_strided_and_unaligned_columns(lm):
    T, ld, E, B = 3001, 19, 13, 1000
    s = synth.qb_scores(T, ld, seed=7)
    hg = lm.qb_histogram(s.cuda(), B, n_cols=E)
    ref = oracle.qb_histogram(s.numpy(), B, n_cols=E)
    assert np.array_equal(hist_np(hg), ref)


def test_histogram_accumulates(lm):
    s = synth.qb_scores(9000, 64, seed=3)
    B = 1000
    hg = lm.qb_histogram(s[:4000].cuda(), B)
    lm.qb_histogram(s[4000:].cuda(), B, hist=hg, accumulate=True)
    assert np.array_equal(hist_np(hg), oracle.qb_histogram(s.numpy(), B))


def test_histogram_overwrites_a_dirty_buffer_then_accumulates(lm):
    """E = 896, B = 1000 (56 groups of 16 experts, a few token chunks each):
    without accumulate every bin is replaced, zeros included, whatever the
    buffer held; with accumulate the counts are added to it."""
    T, E, B = 9000, 896, 1000
    s = synth.qb_scores(T, E, seed=11)
    hg = torch.full((E, B), 0x5A5A5A5A, dtype=torch.int32, device="cuda")   # not zeroed
    lm.qb_histogram(s[:4000].cuda(), B, hist=hg)
    torch.cuda.synchronize()
    assert np.array_equal(hist_np(hg), oracle.qb_histogram(s[:4000].numpy(), B))
    lm.qb_histogram(s[4000:].cuda(), B, hist=hg, accumulate=True)
    torch.cuda.synchronize()
    assert np.array_equal(hist_np(hg), oracle.qb_histogram(s.numpy(), B))


def test_histogram_full_size_sampled(lm):
    """T = 2^20 x 896 (the largest sweep point): every row sums to T and a
    sample of expert columns matches the oracle bit for bit."""
    T, E, B = 1 << 20, 896, 1000
    s = synth.qb_scores(T, E, device="cuda")
    hg = lm.qb_histogram(s, B)
    h = hist_np(hg)
    assert np.all(h.sum(axis=1, dtype=np.uint64) == T)
    cols = np.array([0, 1, 255, 256, 511, 640, 895])
    sub = s[:, torch.from_numpy(cols).cuda()].contiguous().cpu().numpy()
    ref = oracle.qb_histogram(sub, B)
    assert np.array_equal(h[cols], ref)


@pytest.mark.parametrize("B", [10, 1000, 10000])
def test_quantile_bias_matches_oracle(lm, B):
    rng = np.random.default_rng(B)
    E = 896
    hist = rng.integers(0, 50, size=(E, B)).astype(np.uint32)
    hist[3] = 0                                  # empty row
    hist[4] = 0
    hist[4, B - 1] = 7                           # all mass in the last bin
    hist[5] = 0
    hist[5, 0] = 1                               # a single count
    level = 1 - 16 / 896
    hg = torch.from_numpy(hist.view(np.int32)).cuda()
    q, b = lm.qb_quantile_bias(hg, level)
    q_ref, b_ref = oracle.qb_quantile_bias(hist, level)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(b.cpu().numpy(), b_ref)


@pytest.mark.parametrize("B", [1, 2, 3])
def test_histogram_and_quantile_with_very_few_bins(lm, B):
    """B = 1 (every score in one bin: the quantile is the rank's fraction of
    it), B = 2 and 3, with scores on the bin edges (s = k/B) and s = 1.0 (the
    last bin), at the level extremes 0 and 1, one half and 1 - k/E."""
    rng = np.random.default_rng(100 + B)
    T, E = 3001, 40
    s = rng.random((T, E)).astype(np.float32)
    s[:: 7] = np.float32(1.0)
    for j in range(B + 1):
        s[j + 1:: 11, j % E] = np.float32(j / B)
    h = lm.qb_histogram(torch.from_numpy(s).cuda(), B)
    hist = oracle.qb_histogram(s, B)
    assert np.array_equal(h.cpu().numpy().view(np.uint32), hist)
    for level in (0.0, 0.5, 1 - 16 / 896, 1.0):
        q, b = lm.qb_quantile_bias(h, level)
        q_ref, b_ref = oracle.qb_quantile_bias(hist, level)
        assert np.array_equal(q.cpu().numpy(), q_ref), level
        assert np.array_equal(b.cpu().numpy(), b_ref), level


def test_quantile_within_one_bin_of_exact_sort(lm):
    T, E, B = 65536, 896, 1000
    s = synth.qb_scores(T, E, seed=11)
    hg = lm.qb_histogram(s.cuda(), B)
    level = 1 - 16 / 896
    q, _ = lm.qb_quantile_bias(hg, level)
    r = int(np.ceil(level * T))
    exact = torch.kthvalue(s, r, dim=0).values.numpy().astype(np.float64)
    assert np.all(np.abs(q.cpu().numpy() - exact) <= 1.0 / B + 1e-6)


@pytest.mark.parametrize("E", [1, 5, 896, 1500])
def test_sign_update_bit_exact(lm, E):
    rng = np.random.default_rng(E)
    counts = rng.integers(0, 300, E).astype(np.int32)
    counts[: E // 3] = int(np.round(counts.mean()))         # some experts exactly at (or near) the mean
    bias = rng.normal(0, 0.1, E).astype(np.float32)
    got = lm.qb_sign_update(torch.from_numpy(counts).cuda(), 1e-3, torch.from_numpy(bias).cuda())
    assert np.array_equal(got.cpu().numpy(), oracle.sign_update(counts, 1e-3, bias))


@pytest.mark.parametrize("method", ["qb", "sign"])
def test_closed_loop_matches_oracle(lm, method):
    """The balancing loop over a stationary stream of skewed score batches:
    route each batch with the current bias (lmoe_route_static), then update the
    bias by QB (histogram -> quantile -> b = -q) or by the fixed-step rule.
    Loads and biases equal the oracle's bit for bit at every step."""
    T, E, k, n = 4096, 896, 16, 4
    batches = synth.qb_score_stream(T, E, n, seed=3, device="cuda")
    host = batches.cpu().numpy()
    cfg = oracle.LayerConfig(d=64, latent=64, n_experts=E, top_k=k, inter=64, n_shared=1, shared_inter=64)
    b_gpu = torch.zeros(E, dtype=torch.float32, device="cuda")
    b_ref = np.zeros(E, np.float32)
    level = 1 - k / E
    for i in range(n):
        counts_gpu = lm.lmoe_route_static(batches[i], b_gpu, k)["counts"]
        idx_ref, _, _ = oracle.topk(cfg, host[i], b_ref)
        counts_ref = oracle.expert_loads(idx_ref, E)
        assert np.array_equal(counts_gpu.cpu().numpy(), counts_ref), i
        if method == "qb":
            _, b_gpu = lm.qb_quantile_bias(lm.qb_histogram(batches[i], 1000), level)
            _, b_ref = oracle.qb_quantile_bias(oracle.qb_histogram(host[i], 1000), level)
        else:
            lm.qb_sign_update(counts_gpu, 1e-3, b_gpu)
            b_ref = oracle.sign_update(counts_ref, 1e-3, b_ref)
        assert np.array_equal(b_gpu.cpu().numpy(), b_ref), i
