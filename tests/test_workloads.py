"""The seeded input recipes (test_neural_memory_titans_b300/workloads.py) on
the CPU, at small sizes: each recipe draws what its description states (shapes,
dtypes, gate ranges, unit-norm keys, the structure that stands in for the
pages' datasets: an orthogonal key-to-value map, Zipf-distributed codebook
keys, needles re-queried later), the states start where stated, and a seed
reproduces its inputs exactly.  Both the CUDA path's tests and the oracle's
consume these inputs, so a recipe that drifted would change what every parity
test checks."""
import numpy as np
import pytest
import torch

from test_neural_memory_titans_b300 import workloads as W


def _small(wid, **sizes):
    base = dict(B=1, H=2, T=300)
    base.update(sizes)
    if W.WORKLOADS[wid].segment:
        base.setdefault("segment", 0)
    return W.WORKLOADS[wid].with_sizes(**base)


@pytest.mark.parametrize("wid", sorted(W.WORKLOADS))
def test_shapes_dtypes_gate_ranges_and_start_state(wid):
    wl = _small(wid)
    x = W.make_inputs(wl, "cpu", seed=3)
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    for n in ("q", "k", "v"):
        assert x[n].shape == (B, H, T, d) and x[n].dtype == wl.dtype and x[n].is_contiguous()
    for n, (lo, hi) in (("alpha", wl.alpha), ("eta", wl.eta), ("beta", wl.beta)):
        g = x[n]
        assert g.shape == (B, H, T) and g.dtype == torch.float32
        assert float(g.min()) >= lo and float(g.max()) <= hi
        assert float(g.max()) - float(g.min()) > 0.5 * (hi - lo)  # spread over the range, not a constant
    assert x["c"] is None
    assert x["M0"].shape == (B, H, wl.P) and x["S0"].shape == (B, H, wl.P)
    assert torch.count_nonzero(x["S0"]) == 0
    if wl.kind == W.LINEAR:
        assert torch.count_nonzero(x["M0"]) == 0
    else:
        assert abs(float(x["M0"].std()) / wl.w_init_std - 1.0) < 0.05


@pytest.mark.parametrize("wid", sorted(W.WORKLOADS))
def test_keys_and_queries_are_unit_norm(wid):
    x = W.make_inputs(_small(wid), "cpu", seed=4)
    for n in ("q", "k"):
        norms = x[n].float().norm(dim=-1)
        # rounding each element to the input type moves the norm by at most its relative step
        tol = 1e-5 if x[n].dtype == torch.float32 else 2 ** -7
        assert float((norms - 1.0).abs().max()) <= tol, n


def test_linear_d128_values_follow_an_orthogonal_map_plus_noise():
    """v = k R + 0.1 N(0, 1) with R orthogonal per unit: the least-squares map
    from k to v has singular values near 1 (the fit's own error shrinks as
    sqrt(d / T)) and leaves a residual of the noise's size."""
    wl = _small(2, T=16384)
    x = W.make_inputs(wl, "cpu", seed=5)
    for u in range(wl.H):
        k, v = x["k"][0, u].double(), x["v"][0, u].double()
        R = torch.linalg.lstsq(k, v).solution
        s = torch.linalg.svdvals(R)
        assert 0.8 < float(s.min()) and float(s.max()) < 1.2
        assert abs(float((s ** 2).mean()) - 1.0) < 0.05
        assert abs(float((v - k @ R).std()) - 0.1) < 0.005


def test_codebook_keys_are_zipf_and_values_depend_on_the_key_id_only():
    wl = _small(3, H=1, T=40000)
    x = W.make_inputs(wl, "cpu", seed=5)
    ids = x["ids"].reshape(-1)
    assert int(ids.min()) >= 0 and int(ids.max()) < W.CODEBOOK_SIZE
    ranks = torch.arange(1, W.CODEBOOK_SIZE + 1, dtype=torch.float64)
    p = ranks ** -W.ZIPF_S / (ranks ** -W.ZIPF_S).sum()
    freq = torch.bincount(ids, minlength=W.CODEBOOK_SIZE).double() / ids.numel()
    for r in range(3):  # the head of the distribution, within a few standard errors
        se = float((p[r] * (1 - p[r]) / ids.numel()) ** 0.5)
        assert abs(float(freq[r] - p[r])) < 5 * se, r
    # one value per key id: every token of the most frequent id carries the same v
    v = x["v"].reshape(-1, wl.d)
    top = v[ids == int(freq.argmax())]
    assert top.shape[0] > 100 and torch.equal(top, top[:1].expand_as(top))


def test_needle_probes_repeat_an_earlier_key():
    wl = _small(4, H=3, T=4096)
    x = W.make_inputs(wl, "cpu", seed=6)
    pos, probe = x["needles"]
    assert pos.shape == (1, 3, int(wl.T * W.NEEDLE_FRACTION))
    assert bool((probe > pos).all()) and bool((probe < wl.T).all())
    q, k = x["q"], x["k"]
    for u in range(wl.H):
        for p, pr in zip(pos[0, u].tolist(), probe[0, u].tolist()):
            # a probe shared by two needles holds the key of the one placed last: compare with every needle
            # that targets this probe
            sources = [pp for pp, qq in zip(pos[0, u].tolist(), probe[0, u].tolist()) if qq == pr]
            assert any(torch.equal(q[0, u, pr], k[0, u, s]) for s in sources), (u, p, pr)


def test_a_seed_reproduces_its_inputs():
    wl = _small(1)
    a, b = W.make_inputs(wl, "cpu", seed=9), W.make_inputs(wl, "cpu", seed=9)
    c = W.make_inputs(wl, "cpu", seed=10)
    for n in ("q", "k", "v", "alpha", "eta", "beta", "M0"):
        assert torch.equal(a[n], b[n]), n
        assert not torch.equal(a[n], c[n]), n


def test_random_state_scales_with_fan_in():
    wl = _small(1, H=4)
    M, S = W.random_state(wl, "cpu", seed=3, scale=0.5)
    P1 = wl.hidden * wl.d
    for blk, fan_in in ((slice(0, P1), wl.d), (slice(P1, None), wl.hidden)):
        std = np.sqrt(0.5 / fan_in)
        assert abs(float(M[..., blk].std()) / std - 1.0) < 0.03
        assert abs(float(S[..., blk].std()) / (0.1 * std) - 1.0) < 0.03
    ML, SL = W.random_state(_small(2), "cpu", seed=3)
    assert ML.shape == (1, 2, 128 * 128) and abs(float(ML.std()) / np.sqrt(1 / 128) - 1.0) < 0.03
