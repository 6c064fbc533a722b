"""GPU parity of the offline calibration calls (smoothing, transform variants,
K-Means seeding / assignment / update / full training) against the
calibration oracle, through the C ABI."""
import numpy as np
import pytest

from oracle import kmeans_oracle as ko

import torch as t

from vector_quantized_bit_gb300 import _build, _lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    assert t.cuda.is_available(), "GPU tests need a CUDA device"


def dev(a):
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def outlier_keys(n, seed, zero_channel=None):
    r = np.random.default_rng(seed)
    x = r.standard_normal((n, 128))
    for c in r.choice(128, 4, replace=False):
        x[:, c] *= r.uniform(8, 20)
    if zero_channel is not None:
        x[:, zero_channel] = 0.0
    return x.astype(np.float16)


@pytest.mark.parametrize("n", [0, 1, 5, 3000, 70001])
def test_smoothing_is_bit_exact(n):
    x = outlier_keys(max(n, 1), seed=n, zero_channel=7)[:n]
    s = t.empty(128, dtype=t.float32, device="cuda")
    _lib.vqkv_smoothing(dev(x) if n else t.empty((0, 128), dtype=t.float16, device="cuda"), s)
    ref = ko.smoothing_vector(x) if n else np.ones(128, dtype=np.float32)
    assert np.array_equal(s.cpu().numpy(), ref)
    if n:
        xf = (x.astype(np.float32) * 3.5).astype(np.float32)
        _lib.vqkv_smoothing(dev(xf), s)
        assert np.array_equal(s.cpu().numpy(), ko.smoothing_vector(xf))


@pytest.mark.parametrize("variant", ko.VARIANTS)
def test_transform_variants(variant):
    x = outlier_keys(1500, seed=11)
    xd = dev(x)
    out = t.empty((1500, 128), dtype=t.float32, device="cuda")
    s = t.empty(128, dtype=t.float32, device="cuda")
    if variant == "none":
        _lib.vqkv_calib_transform(xd, out)
    elif variant in ("smooth", "smooth_hadamard"):
        _lib.vqkv_smoothing(xd, s)
        _lib.vqkv_calib_transform(xd, out, s_pre=s, rotate=variant == "smooth_hadamard")
    elif variant == "hadamard":
        _lib.vqkv_calib_transform(xd, out, rotate=True)
    else:   # rotate, then smooth the rotated rows by their own factors
        rot = t.empty_like(out)
        _lib.vqkv_calib_transform(xd, rot, rotate=True)
        _lib.vqkv_smoothing(rot, s)
        _lib.vqkv_calib_transform(rot, out, s_post=s)
    ref, s_ref = ko.transform(x, variant)
    if s_ref is not None:
        assert np.allclose(s.cpu().numpy(), s_ref, rtol=2e-7, atol=0)
    got = out.cpu().numpy().astype(np.float64)
    scale = np.abs(ref).max(axis=1, keepdims=True)
    assert (np.abs(got - ref) / scale).max() < 2e-6


def _points(n, dim, seed, dup=False):
    r = np.random.default_rng(seed)
    x = r.standard_normal((n, dim)).astype(np.float32)
    if dup:   # repeated points and ties
        x[n // 2:n // 2 + 40] = x[0]
    return x


@pytest.mark.parametrize("dim,k,n", [(2, 256, 3000), (4, 256, 3000), (8, 300, 2000), (4, 2500, 1500),
                                      (8, 1025, 800), (4, 1, 50)])
def test_assign_matches_oracle(dim, k, n):
    x = _points(n, dim, seed=dim * 7 + k)
    c = _points(k, dim, seed=k + 1)
    if k > 4:
        c[3] = c[1]   # duplicate centroid: its points go to the lower index
    idx = t.empty(n, dtype=t.int32, device="cuda")
    dist = t.empty(n, dtype=t.float32, device="cuda")
    _lib.vqkv_kmeans_assign(dev(x), dev(c), idx, dist)
    got, gd = idx.cpu().numpy(), dist.cpu().numpy()
    ref, d32 = ko.assign(x, c)
    bad = np.nonzero(got != ref)[0]
    assert all(ko.assign_near_tie(d32[i], got[i]) for i in bad), bad[:10]
    assert len(bad) <= max(2, n // 500)
    assert not np.isin(got, [3]).any() or k <= 4
    rel = np.abs(gd.astype(np.float64) - d32[np.arange(n), got]) / np.maximum(d32[np.arange(n), got], 1e-30)
    assert rel.max() < 1e-5


@pytest.mark.parametrize("dim", [2, 4, 8])
def test_update_matches_oracle(dim):
    n, k = 5000, 300
    x = _points(n, dim, seed=dim) * 3
    r = np.random.default_rng(dim + 100)
    a = r.integers(0, k - 20, size=n).astype(np.int32)   # the last 20 clusters are empty
    a[:5] = -1                                            # outside [0, k): no cluster
    a[5:9] = k + 3
    c_in = _points(k, dim, seed=dim + 5)
    c_out = t.empty((k, dim), dtype=t.float32, device="cuda")
    _lib.vqkv_kmeans_update(dev(x), dev(a), dev(c_in), c_out)
    got = c_out.cpu().numpy()
    ref = ko.update(x, a.astype(np.int64), c_in)
    assert np.array_equal(got[k - 20:], c_in[k - 20:])
    ulp = np.spacing(np.abs(ref).astype(np.float32))
    assert (np.abs(got - ref) <= ulp).all()


def _check_seeding(x, u, seeds):
    """Each pick against the oracle's pick from the same earlier picks."""
    n = len(x)
    assert seeds[0] == min(n - 1, int(np.floor(float(u[0]) * n)))
    x64 = x.astype(np.float64)
    d2 = ((x64 - x64[seeds[0]]) ** 2).sum(1)
    ties = 0
    for i in range(1, len(seeds)):
        o = ko.seed_next(d2, u[i])
        if o != seeds[i]:
            assert ko.seed_near_tie(d2, u[i], o, int(seeds[i])), (i, o, seeds[i])
            ties += 1
        d2 = np.minimum(d2, ((x64 - x64[seeds[i]]) ** 2).sum(1))
    return ties


# one CTA (slices in shared memory), clusters of 8 and 16 CTAs, and the
# one-CTA fallback with D^2 in global memory (points beyond 16 slices)
@pytest.mark.parametrize("dim,k,n", [(4, 64, 2000), (8, 200, 3001), (2, 256, 5000), (8, 48, 30000),
                                      (4, 40, 65536), (8, 24, 65536), (8, 16, 100003)])
def test_seeding_matches_oracle(dim, k, n):
    x = _points(n, dim, seed=k, dup=True)
    u = np.random.default_rng(k + n).random(k).astype(np.float32)
    seeds = t.empty(k, dtype=t.int32, device="cuda")
    cent = t.empty((k, dim), dtype=t.float32, device="cuda")
    _lib.vqkv_kmeans_seed(dev(x), dev(u), cent, seeds)
    s = seeds.cpu().numpy()
    ties = _check_seeding(x, u, s)
    assert ties <= 2
    assert np.array_equal(cent.cpu().numpy(), x[s])


def test_seeding_with_identical_points_uses_the_draws():
    x = np.ones((100, 4), dtype=np.float32)
    u = np.array([0.5, 0.0, 0.999, 0.25], dtype=np.float32)
    seeds = t.empty(4, dtype=t.int32, device="cuda")
    cent = t.empty((4, 4), dtype=t.float32, device="cuda")
    _lib.vqkv_kmeans_seed(dev(x), dev(u), cent, seeds)
    assert seeds.cpu().numpy().tolist() == [50, 0, 99, 25]


@pytest.mark.parametrize("dim,k,n,iters", [(4, 128, 4000, 5), (8, 64, 3000, 3), (2, 256, 2000, 0)])
def test_training_is_the_composition_of_the_steps(dim, k, n, iters):
    x = _points(n, dim, seed=n + dim)
    u = np.random.default_rng(iters + 3).random(k).astype(np.float32)
    xd, ud = dev(x), dev(u)
    cent = t.empty((k, dim), dtype=t.float32, device="cuda")
    cb = t.empty((k, dim), dtype=t.float16, device="cuda")
    seeds = t.empty(k, dtype=t.int32, device="cuda")
    last = t.full((n,), -7, dtype=t.int32, device="cuda")
    _lib.vqkv_kmeans(xd, ud, cent, iters, codebook=cb, seeds=seeds, assign=last)
    # the same steps one call at a time, each checked against the oracle
    c = t.empty((k, dim), dtype=t.float32, device="cuda")
    s2 = t.empty(k, dtype=t.int32, device="cuda")
    _lib.vqkv_kmeans_seed(xd, ud, c, s2)
    assert np.array_equal(s2.cpu().numpy(), seeds.cpu().numpy())
    idx = t.empty(n, dtype=t.int32, device="cuda")
    for _ in range(iters):
        _lib.vqkv_kmeans_assign(xd, c, idx)
        ref, d32 = ko.assign(x, c.cpu().numpy())
        got = idx.cpu().numpy()
        assert all(ko.assign_near_tie(d32[i], got[i]) for i in np.nonzero(got != ref)[0])
        nxt = t.empty_like(c)
        _lib.vqkv_kmeans_update(xd, idx, c, nxt)
        ref_c = ko.update(x, got.astype(np.int64), c.cpu().numpy())
        assert (np.abs(nxt.cpu().numpy() - ref_c) <= np.spacing(np.abs(ref_c).astype(np.float32))).all()
        c = nxt
    assert np.array_equal(cent.cpu().numpy(), c.cpu().numpy())
    assert np.array_equal(cb.cpu().numpy(), c.cpu().numpy().astype(np.float16))
    if iters:
        assert np.array_equal(last.cpu().numpy(), idx.cpu().numpy())
    else:
        assert (last.cpu().numpy() == -7).all()
    # deterministic
    cent2 = t.empty_like(cent)
    _lib.vqkv_kmeans(xd, ud, cent2, iters)
    assert t.equal(cent, cent2)


def test_training_recovers_separated_blobs():
    r = np.random.default_rng(21)
    means = r.uniform(-50, 50, size=(32, 8))
    x = np.concatenate([m + r.standard_normal((150, 8)) * 0.3 for m in means]).astype(np.float32)
    u = r.random(32).astype(np.float32)
    cent = t.empty((32, 8), dtype=t.float32, device="cuda")
    _lib.vqkv_kmeans(dev(x), dev(u), cent, 10)
    got = cent.cpu().numpy().astype(np.float64)
    blob = np.stack([x[i * 150:(i + 1) * 150].astype(np.float64).mean(0) for i in range(32)])
    d = ko.squared_distances(blob, got)
    assert (np.sqrt(d.min(axis=1)) < 1e-4).all()
