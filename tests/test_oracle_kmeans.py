"""Pins of the calibration / K-Means oracle (oracle/kmeans_oracle.py) to
facts that do not come from the oracle itself: hand-worked examples, a
library Hadamard, closed forms (means, orthogonality), invariances and the
sampling law of k-means++ (Arthur and Vassilvitskii, 2007)."""
import numpy as np
import pytest
import scipy.linalg

from oracle import kmeans_oracle as ko
from oracle import vqkv_oracle as vo


def test_smoothing_vector_hand_example():
    rows = np.array([[1.0, -4.0, 0.0, 0.25],
                     [-9.0, 2.0, 0.0, -0.5]], dtype=np.float16)
    s = ko.smoothing_vector(rows)
    assert s.dtype == np.float32
    assert np.array_equal(s, np.array([3.0, 2.0, 1.0, np.sqrt(0.5)], dtype=np.float32))


def test_smoothing_vector_ignores_order_and_sign():
    r = np.random.default_rng(1)
    x = r.standard_normal((50, 128)).astype(np.float16)
    s = ko.smoothing_vector(x)
    assert np.array_equal(s, ko.smoothing_vector(-x[::-1]))
    # and it is the per-channel max magnitude's square root, channel by channel
    for c in (0, 17, 127):
        assert s[c] == np.float32(np.sqrt(np.abs(x[:, c].astype(np.float64)).max()))


def test_hadamard_matches_library_and_is_orthogonal():
    h = ko.hadamard(128)
    assert np.array_equal(h * np.sqrt(128), scipy.linalg.hadamard(128).astype(np.float64))
    assert np.abs(h @ h.T - np.eye(128)).max() < 1e-12


@pytest.mark.parametrize("variant", ko.VARIANTS)
def test_transform_round_trip(variant):
    r = np.random.default_rng(2)
    x = (r.standard_normal((20, 128)) * 3).astype(np.float16)
    xt, s = ko.transform(x, variant)
    back = ko.inverse_transform(xt, variant, s)
    assert np.abs(back - x.astype(np.float64)).max() < 1e-12


def test_vecinfer_variant_is_the_decode_path_key_transform():
    r = np.random.default_rng(3)
    x = (r.standard_normal((8, 128)) * 2).astype(np.float16)
    s = ko.smoothing_vector(x)
    xt, _ = ko.transform(x, "smooth_hadamard", s)
    assert np.abs(xt - vo.transform_keys(x, s).astype(np.float64)).max() < 1e-5
    # and by the library rotation
    ref = (x.astype(np.float64) / s.astype(np.float64)) @ (scipy.linalg.hadamard(128) / np.sqrt(128))
    assert np.abs(xt - ref).max() < 1e-12


def test_hadamard_smooth_flattens_the_rotated_maxima():
    """The "order" variant divides the rotated keys by their own smoothing
    vector, so every channel's largest magnitude becomes sqrt of itself."""
    r = np.random.default_rng(4)
    x = r.standard_normal((200, 128)).astype(np.float16)
    xt, s = ko.transform(x, "hadamard_smooth")
    m = np.abs(xt).max(axis=0)
    assert np.allclose(m, s.astype(np.float64), rtol=1e-6)


def test_squared_distances_by_hand_and_expanded_form():
    x = np.array([[0.0, 0.0], [1.0, 2.0]], dtype=np.float32)
    c = np.array([[1.0, 1.0], [3.0, -1.0]], dtype=np.float32)
    assert np.array_equal(ko.squared_distances(x, c), np.array([[2.0, 10.0], [1.0, 13.0]]))
    r = np.random.default_rng(5)
    x = r.standard_normal((40, 8)).astype(np.float32)
    c = r.standard_normal((30, 8)).astype(np.float32)
    x64, c64 = x.astype(np.float64), c.astype(np.float64)
    expanded = (x64 ** 2).sum(1)[:, None] - 2 * x64 @ c64.T + (c64 ** 2).sum(1)[None, :]
    assert np.abs(ko.squared_distances(x, c) - expanded).max() < 1e-10


def test_assign_ties_to_lowest_index_and_exact_centroid():
    c = np.array([[0.0, 0.0], [2.0, 0.0], [2.0, 0.0], [5.0, 5.0]], dtype=np.float32)
    x = np.array([[1.0, 0.0],     # equidistant from 0, 1, 2 -> 0
                  [2.0, 0.0],     # exactly centroid 1 (and 2) -> 1
                  [4.0, 4.0]], dtype=np.float32)
    idx, d32 = ko.assign(x, c)
    assert list(idx) == [0, 1, 3]
    assert d32[1, 1] == 0.0
    assert ko.assign_near_tie(d32[0], 1) and not ko.assign_near_tie(d32[2], 0)


def test_update_is_the_mean_and_empty_clusters_stay():
    x = np.array([[0.0, 0.0], [2.0, 4.0], [10.0, 10.0], [11.0, 13.0], [12.0, 10.0]], dtype=np.float32)
    idx = np.array([0, 0, 2, 2, 2])
    c = np.array([[9.0, 9.0], [-1.0, -1.0], [0.0, 0.0]], dtype=np.float32)
    out = ko.update(x, idx, c)
    assert np.array_equal(out, np.array([[1.0, 2.0], [-1.0, -1.0], [11.0, 11.0]], dtype=np.float32))
    perm = np.random.default_rng(6).permutation(5)
    assert np.array_equal(ko.update(x[perm], idx[perm], c), out)


def test_seed_next_by_hand():
    d2 = np.array([0.0, 1.0, 3.0])
    assert ko.seed_next(d2, 0.5) == 2          # threshold 2: running sums 0, 1, 4
    assert ko.seed_next(d2, 0.0) == 1          # a chosen point (D^2 = 0) is never drawn
    assert ko.seed_next(d2, 0.2499) == 1       # threshold just under 1
    assert ko.seed_next(d2, 0.25) == 2         # running sum must exceed the threshold
    assert ko.seed_next(np.zeros(4), 0.74) == 2   # all zero: floor(u * n)
    assert ko.seed_near_tie(d2, 0.25, 1, 2) and not ko.seed_near_tie(d2, 0.5, 1, 2)


def test_seed_next_samples_in_proportion_to_d2():
    d2 = np.array([1.0, 0.0, 2.0, 5.0, 0.0, 2.0])
    u = (np.arange(100000) + 0.5) / 100000
    picks = np.array([ko.seed_next(d2, x) for x in u[::10]])
    freq = np.bincount(picks, minlength=6) / len(picks)
    assert np.abs(freq - d2 / d2.sum()).max() < 2e-3


def test_seed_puts_one_centre_in_each_separated_blob():
    r = np.random.default_rng(7)
    centres = np.array([[0, 0], [100, 0], [0, 100], [100, 100], [50, 300]], dtype=np.float64)
    x = np.concatenate([c + r.standard_normal((40, 2)) for c in centres]).astype(np.float32)
    u = r.random(5)
    chosen = ko.seed(x, 5, u)
    assert sorted(set((chosen // 40).tolist())) == [0, 1, 2, 3, 4]
    assert chosen[0] == int(np.floor(u[0] * len(x)))


def test_seed_with_k_equal_n_picks_every_distinct_point():
    r = np.random.default_rng(8)
    x = r.standard_normal((12, 3)).astype(np.float32)
    chosen = ko.seed(x, 12, r.random(12))
    assert sorted(chosen.tolist()) == list(range(12))


def test_seed_d2_against_the_incremental_minimum():
    r = np.random.default_rng(9)
    x = r.standard_normal((30, 4)).astype(np.float32)
    chosen = [3, 17, 5]
    d2 = ko.seed_d2(x, chosen)
    ref = np.min([((x.astype(np.float64) - x[c].astype(np.float64)) ** 2).sum(1) for c in chosen], axis=0)
    assert np.array_equal(d2, ref)


def test_kmeans_recovers_separated_blob_means():
    r = np.random.default_rng(10)
    means = np.array([[0, 0, 0, 0], [20, 0, 0, 0], [0, 20, 0, 0], [0, 0, 20, 0]], dtype=np.float64)
    x = np.concatenate([m + r.standard_normal((100, 4)) * 0.5 for m in means]).astype(np.float32)
    c, cb = ko.kmeans(x, 4, 5, r.random(4))
    order = np.argsort(c[:, 0] + 2 * c[:, 1] + 4 * c[:, 2])
    blob_means = np.stack([x[i * 100:(i + 1) * 100].astype(np.float64).mean(0) for i in range(4)])
    assert np.abs(c[order] - blob_means).max() < 1e-5
    assert cb.dtype == np.float16 and np.array_equal(cb, c.astype(np.float16))


def test_kmeans_single_centroid_is_the_global_mean():
    r = np.random.default_rng(11)
    x = r.standard_normal((300, 8)).astype(np.float32)
    c, _ = ko.kmeans(x, 1, 1, np.array([0.3]))
    assert np.abs(c[0] - x.astype(np.float64).mean(0)).max() < 1e-6


def test_lloyd_objective_never_increases():
    r = np.random.default_rng(12)
    x = r.standard_normal((500, 4)).astype(np.float32)
    c = x[ko.seed(x, 16, r.random(16))].copy()
    prev = ko.objective(x, c)
    for _ in range(6):
        idx, _ = ko.assign(x, c)
        c = ko.update(x, idx, c)
        cur = ko.objective(x, c)
        assert cur <= prev + 1e-12
        prev = cur


def test_relative_error_and_utilization_by_hand():
    x = np.array([[3.0, 4.0]])
    assert ko.relative_error(x, np.array([[3.0, 3.0]])) == pytest.approx(1.0 / 25.0)
    frac, ent = ko.utilization(np.array([0, 0, 1, 3]), 4)
    assert frac == 0.75
    assert ent == pytest.approx(1.5)
