"""The seeded workload definitions: which key channels are scaled up, and
which workloads build dense-and-sparse caches.  No GPU needed."""

import numpy as np

from bit_kv_cache_02_gb300 import synth


def test_fixed_outlier_channels_only_where_a_workload_lists_them():
    tiny = synth.WORKLOADS["tiny"]
    oc = synth.outlier_channels(tiny, 0)
    assert oc.shape == (1, 4) and oc.tolist() == [[3, 17, 64, 101]]
    assert not tiny.dense_sparse


def test_drawn_outlier_channels_differ_per_head_and_layer():
    """Four distinct channels per (layer, KV head) drawn from the seed; the
    dense-and-sparse workload uses the same draw as the plain one."""
    for name in ("llama2_7b_mha", "llama2_7b_mha_outliers"):
        w = synth.WORKLOADS[name]
        oc = synth.outlier_channels(w, 0)
        assert oc.shape == (w.kv_heads, 4)
        assert all(len(set(row)) == 4 for row in oc.tolist())
        assert len({tuple(sorted(row)) for row in oc.tolist()}) > w.kv_heads // 2
        assert (oc >= 0).all() and (oc < 128).all()
        assert not np.array_equal(oc, synth.outlier_channels(w, 1))
    np.testing.assert_array_equal(synth.outlier_channels(synth.WORKLOADS["llama2_7b_mha"], 3),
                                  synth.outlier_channels(synth.WORKLOADS["llama2_7b_mha_outliers"], 3))


def test_dense_sparse_flag_is_set_only_on_its_workload():
    flagged = sorted(n for n, w in synth.WORKLOADS.items() if w.dense_sparse)
    assert flagged == ["llama2_7b_mha_outliers"]


def test_outlier_channels_scale_the_drawn_keys():
    w = synth.WORKLOADS["llama2_7b_mha"]
    small = synth.Workload("small", 1, 2, 4, 4, 64, 2)
    k, v = synth.kv_tokens(small, 0, 64)
    oc = synth.outlier_channels(small, 0)
    kk = k.float().abs().mean(dim=(0, 2)).numpy()        # [heads][channels]
    for h in range(4):
        others = np.setdiff1d(np.arange(128), oc[h])
        assert kk[h, oc[h]].min() > 5 * kk[h, others].max()
    assert w.outlier_mult == 15.0
