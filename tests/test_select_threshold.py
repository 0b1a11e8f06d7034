"""The selector's float threshold test is the image test.

The top-16 selector ranks 64-bit keys whose upper half is the
order-preserving image of a score: NaN ranked as -inf, -0 as +0, then the
sign-magnitude bits flipped so that unsigned order is score order ("wolfcomos/
MSA PR #1", Changes; "vllm ... indexer_nvfp4_decode_cp", _page_keys).  The
kernel keeps the scores as floats, takes each lane's maximum with fmaxf, and
lets a score survive when it compares >= the float whose image is the
threshold, whenever the threshold lies above the image of -inf.  These
host-side checks restate the image map from its definition and confirm, on
every special value and on random floats, that

  * the image of fmaxf over a lane equals the largest image of the lane;
  * for every threshold above image(-inf), (x >= t) == (image(x) >= thr),
    t being the float the inverse map gives for thr (NaN never survives,
    -0 and +0 compare equal);

so the float pass selects exactly the survivors of the image pass.
"""

import numpy as np


def image(x: np.ndarray) -> np.ndarray:
    """Order-preserving 32-bit image, written from the key's definition."""
    x = np.asarray(x, dtype=np.float32).copy()
    x[np.isnan(x)] = -np.inf  # NaN ranks as -inf
    x[x == 0] = np.float32(0.0)  # -0 ranks as +0
    b = x.view(np.uint32).astype(np.uint64)
    neg = (b >> 31) == 1
    out = np.where(neg, (~b) & 0xFFFFFFFF, b ^ 0x80000000)
    return out.astype(np.uint64)


def inverse(thr: np.ndarray) -> np.ndarray:
    """The float whose image is thr (thr an image of a canonical score)."""
    thr = np.asarray(thr, dtype=np.uint64)
    bits = np.where(thr & 0x80000000, thr ^ 0x80000000, (~thr) & 0xFFFFFFFF)
    return bits.astype(np.uint32).view(np.float32)


def specials():
    f = np.finfo(np.float32)
    return np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, f.max, -f.max, f.tiny, -f.tiny,
                     np.float32(1e-45), np.float32(-1e-45), 1.0, -1.0, 0.5, -0.5, 448.0, -448.0],
                     dtype=np.float32)


def test_image_is_order_preserving():
    rng = np.random.default_rng(0)
    x = np.concatenate([specials(), rng.standard_normal(4000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e30).astype(np.float32)])
    canon = x.copy()
    canon[np.isnan(canon)] = -np.inf
    ix = image(x)
    # unsigned order of images == float order of the canonical scores
    i, j = rng.integers(0, len(x), size=(2, 20000))
    assert np.array_equal(ix[i] > ix[j], canon[i] > canon[j])
    assert np.array_equal(ix[i] == ix[j], canon[i] == canon[j])
    # every real score's image is above 0 (0 marks "no column")
    assert (ix > 0).all()


def test_lane_max_by_fmaxf_has_the_largest_image():
    rng = np.random.default_rng(1)
    pool = np.concatenate([specials(), rng.standard_normal(64).astype(np.float32)])
    for _ in range(3000):
        lane = rng.choice(pool, size=rng.integers(1, 12))
        m = np.float32(np.nan)
        for v in lane:
            m = np.fmax(m, v)  # fmaxf: a NaN operand yields the other one
        assert image(np.array([m]))[0] == image(lane).max()


def test_float_compare_equals_image_compare_above_neg_inf():
    rng = np.random.default_rng(2)
    x = np.concatenate([specials(), rng.standard_normal(3000).astype(np.float32),
                        rng.choice(np.array([0.0, -0.0, 1.0, -1.0], dtype=np.float32), 500)])
    neg_inf_image = image(np.array([-np.inf], dtype=np.float32))[0]
    # thresholds: images of real scores strictly above the image of -inf
    cand = image(np.concatenate([specials(), rng.standard_normal(300).astype(np.float32)]))
    thrs = np.unique(cand[cand > neg_inf_image])
    ix = image(x)
    with np.errstate(invalid="ignore"):
        for thr in thrs:
            t = inverse(np.array([thr]))[0]
            assert image(np.array([t]))[0] == thr  # the inverse is exact
            assert np.array_equal(x >= t, ix >= thr), (thr, t)
