"""The seeded input generators: reproducible, bf16-exact, and built as the recipes say."""
import numpy as np

import workloads as W


def test_slices_are_reproducible_and_independent():
    w = W.GPT2_LAYER
    a = W.slice_inputs(w, 1, 3)
    b = W.slice_inputs(w, 1, 3)
    c = W.slice_inputs(w, 1, 4)
    for n in W.TENSORS:
        assert np.array_equal(a[n], b[n])
        assert not np.array_equal(a[n], c[n])
    assert not np.array_equal(a["Q"], a["K"])


def test_bf16_inputs_are_exactly_representable():
    import torch
    x = W.slice_inputs(W.GPT2_LAYER, 0, 0)["Q"]
    t = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(t, x)
    # and the rounding is torch's RNE of the raw draws
    raw = W._normal(W.GPT2_LAYER, "Q", 0, 0)
    assert np.array_equal(torch.from_numpy(raw).to(torch.bfloat16).float().numpy(), x)


def test_f32_inputs_are_raw_normals():
    x = W.slice_inputs(W.TINY_F32, 0, 0)
    assert x["Q"].dtype == np.float32 and x["Q"].shape == (256, 64)
    assert abs(float(x["Q"].std()) - 1.0) < 0.03


def test_full_day_dO_scale():
    s = W.slice_inputs(W.FULL_DAY.with_n(4096), 0, 0, ("dO", "Q"))
    assert abs(float(s["dO"].std()) - 0.1) < 0.005 and abs(float(s["Q"].std()) - 1.0) < 0.05


def test_large_key_construction():
    w = W.LARGE_KEY.with_n(512)
    s0 = W.slice_inputs(w, 0, 2, ("Q", "K"))
    s1 = W.slice_inputs(w, 5, 2, ("Q", "K"))
    # shared per-head mean of norm 40 (same head, different batch)
    m0, m1 = s0["K"].mean(axis=0), s1["K"].mean(axis=0)
    assert abs(np.linalg.norm(m0) - 40) < 2.5 and np.linalg.norm(m0 - m1) < 4
    # each query (i >= 1) is close to half of some earlier key
    K, Q = s0["K"].astype(np.float64), s0["Q"].astype(np.float64)
    for i in (1, 7, 300, 511):
        dist = np.linalg.norm(Q[i][None, :] - 0.5 * K[:i], axis=1)
        assert dist.min() < 0.5 * np.sqrt(w.d) * 1.5
    assert s0["Q"].dtype == np.float32


def test_workload_table():
    assert W.GPT2_LAYER.rows == 4 * 12 * 1024
    assert [w.N for w in W.LONG_SWEEP] == [4096, 16384, 65536, 262144]
    assert W.FULL_DAY.N % 128 == 104
    assert W.LARGE_KEY.d == 128 and abs(W.LARGE_KEY.scale - 128 ** -0.5) < 1e-15


def test_grouped_heads_draw_key_side_tensors_per_key_value_head():
    w = W.Workload("gqa", 2, 6, 9, 8, "bf16", group=3)
    x = W.inputs(w)
    for n in W.TENSORS:
        assert x[n].shape == (2, 2 if n in W.KV_TENSORS else 6, 9, 8), n
    plain = W.inputs(W.Workload("gqa", 2, 6, 9, 8, "bf16"))
    for n in W.TENSORS:  # the same per-slice streams as the ungrouped workload
        k = x[n].shape[1]
        assert np.array_equal(x[n], plain[n][:, :k])
    import pytest
    with pytest.raises(ValueError):
        W.inputs(w, heads=[0])


def test_segment_ids_are_runs_of_the_stated_lengths():
    s = W.segment_ids(3, 5000, 64, seed=1)
    assert s.shape == (3, 5000) and s.dtype == np.int32
    assert np.all(np.diff(s, axis=1) >= 0) and np.all(s[:, 0] == 0)
    for b in range(3):
        lens = np.bincount(s[b])
        assert np.all(lens[:-1] >= 1) and np.all(lens[:-1] <= 127) and 40 < lens[:-1].mean() < 90
    assert np.array_equal(s, W.segment_ids(3, 5000, 64, seed=1))
    assert not np.array_equal(s[0], s[1])
