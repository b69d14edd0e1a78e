"""The seeded input generator: known-answer vectors, determinism, recipe shape."""
import numpy as np
import pytest

import workloads as W


def test_philox_known_answers():
    # Known-answer vectors published with the Random123 reference implementation
    # of Philox4x32-10 (Salmon et al., SC'11).
    assert W.philox_kat([0, 0, 0, 0], [0, 0]).tolist() == [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]
    assert W.philox_kat([0xffffffff] * 4, [0xffffffff] * 2).tolist() == [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]
    assert W.philox_kat([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344],
                        [0xa4093822, 0x299f31d0]).tolist() == [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1]


def test_rows_regenerate_independently():
    w = W.get("confident_bf16").with_shape(64, 1003)
    full = w.logits_rows(0, 64)
    part = w.logits_rows(17, 5)
    assert np.array_equal(full[17:22], part)
    assert np.array_equal(full, w.logits_rows(0, 64))


def test_distribution_and_counts():
    w = W.get("ce_z_bf16")
    x = w.logits_rows(0, 64)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(f.mean()) < 0.01 and abs(f.std() - 3.0) < 0.01
    t = w.targets()
    assert (t == -100).sum() == 410
    assert t[t >= 0].max() < w.V
    w1 = W.get("ce_fp32_small")
    assert (w1.targets() == -100).sum() == 6 and w1.n_active() == 58
    assert np.isfinite(w1.margins()).sum() == 8
    w5 = W.get("ce_z_kl_bf16")
    assert (w5.loss_mask() == 0).sum() == 3277


def test_planted_margins():
    w = W.get("ce_fp32_small")
    t = w.targets()
    m = w.margins()
    z = w.logits_rows(0, w.T).astype(np.float64)
    for r in np.where(np.isfinite(m))[0]:
        assert t[r] >= 0
        others = np.delete(z[r], t[r])
        assert z[r, t[r]] - others.max() == pytest.approx(m[r], abs=1e-5)
    assert sorted(set(m[np.isfinite(m)].tolist())) == [20.0, 30.0]


def test_teacher_is_student_plus_noise():
    w = W.get("ce_z_kl_bf16").with_shape(8, 4096)
    s = w.logits_rows(0, 8)
    u = w.teacher_rows(0, 8, s)
    d = (u.astype(np.uint32) << 16).view(np.float32) - (s.astype(np.uint32) << 16).view(np.float32)
    assert abs(d.std() - 1.0) < 0.05


def test_gspo_segments():
    w = W.get("gspo_z_bf16")
    seg, S, adv = w.segments()
    assert seg.min() == 0 and seg.max() == S - 1
    # ids are contiguous runs, non-decreasing, none straddles a packed row
    assert np.all(np.diff(seg) >= 0)
    for p in range(w.T // w.packed_len):
        blk = seg[p * w.packed_len:(p + 1) * w.packed_len]
        k = len(np.unique(blk))
        assert 1 <= k <= 64
    assert adv.shape == (S,)
