"""GPU parity of top-k temperature sampling (ds4f-disk issue #6, work item 3
and step 3: the head's logits feed top-k / temperature sampling, a softmax
sampler driven by a seeded generator).

The selection is exact: the k rows and their order must equal the float64
oracle's on the same float32 logits, and top_value must be those logits bit
for bit.  Probabilities are float32 (expf within 2 ulp), checked against the
oracle within a bound derived from that arithmetic; the token must be the
oracle's, or lie across a boundary that u * S falls within rounding of.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_weight_matvec_gb300 import qmv, synth

pytestmark = pytest.mark.gpu

EPS = 2.0 ** -24
TINY = 2.0 ** -126


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qmv.load()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def logits(seed, batch, R, kind="normal"):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return (rng.standard_normal((batch, R)) * 3).astype(np.float32)
    if kind == "ties":
        return rng.integers(-6, 7, (batch, R)).astype(np.float32)
    if kind == "equal":
        return np.full((batch, R), 0.25, np.float32)
    y = (rng.standard_normal((batch, R)) * 3).astype(np.float32)  # "special"
    for v in range(batch):
        y[v, rng.integers(0, R, 3)] = -0.0
        y[v, rng.integers(0, R, 2)] = -np.inf
        if v % 3 == 1:
            y[v, rng.integers(0, R, 2)] = np.nan
        if v % 3 == 2:
            y[v, rng.integers(0, R, 3)] = np.inf
    return y


def bounds(l, T):
    """Per-entry bound on |p_gpu - p| and the bound on the cumulative sums,
    from the float32 steps: d = l - l0 and a = d / T each rounded (relative
    2^-24, entering the exponent as |a| 2^-23), expf within 2 ulp (2^-22),
    k - 1 rounded additions for S and the cumulative sums, one rounded
    product u * S and one rounded division w / S; doubled.  Weights and
    probabilities below float32's normal range (2^-126) carry an absolute
    error up to that size (gradual underflow, then 0)."""
    a = (l - l[0]) / T
    w = np.exp(a)
    S = w.sum()
    e = w * (np.abs(a) * 2 * EPS + 4 * EPS) + TINY
    dS = e.sum() + len(l) * EPS * S
    p = w / S
    return 2 * (e / S + p * dS / S + p * EPS + TINY), 2 * (dS + S * EPS), w, S


def check(y, k, T, u, got):
    idx, val, prob, tok = (t.cpu().numpy() for t in got)
    ref_idx, ref_prob, ref_tok = oracle.topk_sample(y, k, T, u)
    assert np.array_equal(idx, ref_idx)
    assert np.array_equal(val.view(np.uint32), np.take_along_axis(y, idx, 1).view(np.uint32))
    for v in range(y.shape[0]):
        l = y[v, idx[v]].astype(np.float64)
        if np.isnan(l[0]) or T == 0:
            assert tok[v] == ref_tok[v] == idx[v, 0]
            if np.isnan(l[0]):
                assert np.isnan(prob[v]).all()
            else:
                assert prob[v, 0] == 1.0 and not prob[v, 1:].any()
            continue
        if not np.isfinite(l[0]):
            assert tok[v] == ref_tok[v]
            assert np.array_equal(prob[v], ref_prob[v].astype(np.float32))
            continue
        pb, cb, w, S = bounds(l, T)
        assert np.all(np.abs(prob[v] - ref_prob[v]) <= pb), (v, np.abs(prob[v] - ref_prob[v]).max())
        if tok[v] != ref_tok[v]:
            uu = min(max(float(u[v]), 0.0), 1.0) if not np.isnan(u[v]) else 0.0
            j = int(np.where(idx[v] == tok[v])[0][0])
            jr = int(np.where(idx[v] == ref_tok[v])[0][0])
            c = np.cumsum(w)
            edge = c[min(j, jr)]  # the boundary between the two picks
            assert abs(edge - uu * S) <= cb, (v, j, jr, edge, uu * S, cb)
            assert abs(j - jr) == 1


def run(y, k, T, u):
    got = qmv.topk_sample_t(dev(y), k, T, dev(np.asarray(u, np.float32)))
    torch.cuda.synchronize()
    return got


@pytest.mark.parametrize("R", [1, 5, 64, 4095, 4096, 4097, 10000, 65537, 245760])
@pytest.mark.parametrize("batch,k", [(1, 1), (3, 7), (8, 64)])
def test_topk_shapes(R, batch, k):
    if k > R:
        k = R
    y = logits(R + batch + k, batch, R)
    u = np.random.default_rng(R).random(batch).astype(np.float32)
    check(y, k, 0.8, u, run(y, k, 0.8, u))


@pytest.mark.parametrize("kind", ["ties", "equal", "special"])
@pytest.mark.parametrize("R", [100, 9000, 245760])
def test_topk_ties_and_nonfinite(kind, R):
    batch, k = 6, 64 if R >= 64 else R
    y = logits(R + len(kind), batch, R, kind)
    u = np.random.default_rng(7).random(batch).astype(np.float32)
    check(y, k, 1.0, u, run(y, k, 1.0, u))


@pytest.mark.parametrize("T", [0.0, 1e-3, 0.25, 1.0, 4.0, 100.0])
def test_topk_temperatures(T):
    y = logits(11, 4, 50000)
    u = np.array([0.0, 0.31, 0.77, 0.999], np.float32)
    check(y, 50, T, u, run(y, 50, T, u))


def test_topk_u_clamping():
    y = logits(12, 6, 3000)
    u = np.array([-0.5, 0.0, np.nan, 1.0, 7.0, np.inf], np.float32)
    got = run(y, 10, 1.0, u)
    check(y, 10, 1.0, u, got)
    idx, _, _, tok = (t.cpu().numpy() for t in got)
    assert tok[0] == idx[0, 0] and tok[1] == idx[1, 0] and tok[2] == idx[2, 0]


def test_topk_u_grid_frequencies():
    """A grid of u over one vector reproduces the probabilities."""
    N, k = 4000, 16
    y = np.tile(logits(13, 1, 20000), (8, 1))
    tokens = []
    for s in range(0, N, 8):
        u = ((np.arange(s, s + 8) + 0.5) / N).astype(np.float32)
        idx, _, prob, tok = (t.cpu().numpy() for t in run(y, k, 0.5, u))
        tokens.extend(tok.tolist())
    counts = np.array([tokens.count(int(i)) for i in idx[0]])
    assert counts.sum() == N
    assert np.all(np.abs(counts - N * prob[0].astype(np.float64)) <= 1.0 + N * 1e-5)


def test_topk_independent_of_slicing():
    """Large R: batch 8 runs 128 slices per vector, batch 1 runs 1024; the
    results are the same."""
    R, k = 1 << 22, 32
    y = logits(14, 8, R)
    u = np.random.default_rng(14).random(8).astype(np.float32)
    many = [t.cpu().numpy() for t in run(y, k, 0.9, u)]
    for v in (0, 5):
        one = [t.cpu().numpy() for t in run(y[v:v + 1], k, 0.9, u[v:v + 1])]
        for a, b in zip(many, one):
            assert np.array_equal(a[v:v + 1].view(np.uint8), b[:1].view(np.uint8))
    check(y[:2], k, 0.9, u[:2], [torch.from_numpy(t[:2]) for t in many])


def test_topk_deterministic():
    y = logits(15, 8, 245760)
    u = np.random.default_rng(15).random(8).astype(np.float32)
    a = [t.cpu().numpy() for t in run(y, 64, 1.0, u)]
    b = [t.cpu().numpy() for t in run(y, 64, 1.0, u)]
    for p, q in zip(a, b):
        assert np.array_equal(p.view(np.uint8), q.view(np.uint8))


@pytest.fixture(scope="module")
def head():
    f = synth.f8_inputs(5, 245760, 4096, 1920, 32, 118, 132, batch=8)
    return f, dev(f.w), dev(f.scale)


@pytest.mark.parametrize("batch", [1, 4, 8])
def test_f8_head_topk_sample(head, batch):
    """The fused call on the 245760 x 4096 head: y is f8_matvec's output bit
    for bit (checked against the oracle on sampled rows) and the sampler
    works on exactly that y."""
    f, w, s = head
    xs = np.ascontiguousarray(f.x[:batch])
    x = dev(xs)
    u = np.random.default_rng(batch).random(batch).astype(np.float32)
    y, idx, val, prob, tok = qmv.f8_matvec_topk_sample_t(w, s, x, 64, 1.0, dev(u))
    y_plain = qmv.f8_matvec_t(w, s, x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y_plain.view(torch.int32))
    yh = y.cpu().numpy()
    check(yh, 64, 1.0, u, (idx, val, prob, tok))
    rows = np.unique(np.concatenate([idx.cpu().numpy().ravel(), np.arange(0, 245760, 4099)]))
    for r in rows[:200]:
        ref, mag = oracle.f8_matvec(f.w, f.scale, xs, rows=(int(r), int(r) + 1))
        assert np.all(np.abs(yh[:, r] - ref[:, r]) <= 1e-4 * mag[:, r] + 1e-6)


def test_f8_head_topk_greedy_matches_argmax():
    f = synth.f8_inputs(6, 20000, 1024, 40, 8, 118, 132, batch=3)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    u = dev(np.array([0.2, 0.5, 0.9], np.float32))
    y, idx, val, prob, tok = qmv.f8_matvec_topk_sample_t(w, s, x, 8, 0.0, u)
    am_idx, am_val = qmv.f8_matvec_argmax_t(w, s, x)
    torch.cuda.synchronize()
    assert torch.equal(tok, am_idx)
    assert torch.equal(val[:, 0], am_val)


@pytest.mark.parametrize("batch", [1, 4, 8])
def test_i8_head_topk_sample(batch):
    """The I8 head (245760 x 4096, per-16 E8M0 group scales) then sampling,
    the token loop of the I8 head: y is i8_matvec's output bit for bit and
    the sampler works on exactly that y."""
    f = synth.i8_inputs(7, 245760, 4096, 110, 124, batch=batch)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    u = np.random.default_rng(batch + 10).random(batch).astype(np.float32)
    y, idx, val, prob, tok = qmv.i8_matvec_topk_sample_t(w, s, x, 64, 0.7, dev(u))
    y_plain = qmv.i8_matvec_t(w, s, x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y_plain.view(torch.int32))
    yh = y.cpu().numpy()
    check(yh, 64, 0.7, u, (idx, val, prob, tok))
    for r in np.unique(idx.cpu().numpy().ravel())[:64]:
        ref, mag = oracle.i8_matvec(f.w, f.scale, f.x, rows=(int(r), int(r) + 1))
        assert np.all(np.abs(yh[:, r] - ref[:, r]) <= 1e-4 * mag[:, r] + 1e-6)


@pytest.mark.parametrize("R,k", [(64, 64), (65, 64), (4096, 64), (4160, 64), (8192, 33)])
def test_topk_k_near_R_and_tile_edges(R, k):
    """k equal to R, one row more than k, and R at and just past the
    4096-entry tile (one slice, then two slices with a ragged second)."""
    y = logits(R * 7 + k, 3, R, "ties")
    u = np.array([0.05, 0.5, 0.95], np.float32)
    check(y, k, 0.6, u, run(y, k, 0.6, u))


@pytest.mark.parametrize("batch", [2, 3, 5])
def test_f8_topk_sample_tensor_core_batches(batch):
    """The fused call where the head runs on the tensor-core kernels with a
    partly used vector group (batch 3, 5)."""
    f = synth.f8_inputs(9, 20000, 1024, 40, 8, 118, 132, batch=batch)
    w, s, x = dev(f.w), dev(f.scale), dev(f.x)
    u = np.random.default_rng(batch + 20).random(batch).astype(np.float32)
    y, idx, val, prob, tok = qmv.f8_matvec_topk_sample_t(w, s, x, 16, 1.5, dev(u))
    y_plain = qmv.f8_matvec_t(w, s, x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y_plain.view(torch.int32))
    yh = y.cpu().numpy()
    check(yh, 16, 1.5, u, (idx, val, prob, tok))
    ref, mag = oracle.f8_matvec(f.w, f.scale, f.x)
    assert np.all(np.abs(yh - ref) <= 1e-4 * mag + 1e-6)
