"""Host-side arithmetic of bench.py: the algorithmic byte counts behind the
roofline, the decode state the timing runs on, and the gate that keeps a
stale ncu summary from supplying the traffic figure.  No GPU needed."""

import os

import numpy as np

import bench
import oracle
from bit_kv_cache_02_gb300 import synth


def test_decode_bytes_count_blocks_window_query_and_output():
    """Per (sequence, KV head): every packed group block once, every fp16
    sink and window token of K and V once; per (sequence, query head): the
    query and the output row."""
    w = synth.WORKLOADS["llama2_7b_mha"]
    bb = oracle.block_bytes(2)
    L = 4097                            # 4096 quantized tokens, one in the window
    want = 16 * 32 * (4096 // 32 * bb + 1 * 2 * 128 * 2) + 16 * 32 * 128 * 2 * 2
    assert bench.decode_bytes(np.full(16, L), w) == want
    assert bench.decode_bytes(np.full(16, L), w) == 218628096
    ws = synth.WORKLOADS["kvquant_prerope"]   # a sink token: 16385 = 1 + 16384 quantized
    assert bench.decode_bytes(np.full(8, 16385), ws) == \
        8 * 32 * (16384 // 32 * bb + 1 * 2 * 128 * 2) + 8 * 32 * 128 * 2 * 2


def test_decode_bytes_follow_the_block_layout_of_each_option():
    for name, kpt, sp in (("llama2_7b_mha_key_per_token", True, False), ("llama2_7b_mha_outliers", False, True)):
        w = synth.WORKLOADS[name]
        bb = oracle.block_bytes(2, key_per_token=kpt, outliers=sp)
        assert bench.decode_bytes(np.full(16, 4097), w) == 16 * 32 * (128 * bb + 512) + 16 * 32 * 512


def test_prefill_bytes_read_fp16_and_write_blocks():
    """Quantized tokens read 512 B of fp16 K and V per token-head and write
    their share of a block; window tokens are read and written as fp16."""
    w = synth.WORKLOADS["llama2_7b_mha"]
    L = 4090                            # 3968 quantized, 122 in the window
    want = 16 * 32 * (3968 * (512 + oracle.block_bytes(2) // 32) + 122 * 2 * 512)
    assert bench.prefill_bytes(np.full(16, L), w) == want


def test_decode_is_timed_on_the_workloads_own_state():
    """After the untimed steps the cache holds context + 1 tokens per
    sequence: for the Llama-2 shape 4096 quantized tokens and a one-token
    window, as the configuration states."""
    for name in ("llama2_7b_mha", "llama3_8b_gqa_2bit", "long_1m", "kvquant_prerope"):
        w = synth.WORKLOADS[name]
        untimed = 9
        pre = bench.prefill_lengths(w, untimed)
        assert (pre + untimed == synth.context_lengths(w) + 1).all()
    w = synth.WORKLOADS["llama2_7b_mha"]
    n = int(bench.prefill_lengths(w, 9)[0]) + 9 - w.num_sink
    assert n % w.residual == 1


def test_stale_profiles_give_no_traffic(tmp_path, monkeypatch):
    """The traffic figure comes from a committed ncu summary only while its
    recorded source hash matches the kernel source."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    good = bench.kernel_source_hash()
    (prof / "a.md").write_text(f"traffic_per_algorithmic_byte: 1.02 source_hash: {good}\n")
    (prof / "b.md").write_text("traffic_per_algorithmic_byte: 1.02 source_hash: 0123456789abcdef\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    real = os.path.join(os.path.dirname(bench.__file__), "bit_kv_cache_02_gb300")
    os.symlink(real, tmp_path / "bit_kv_cache_02_gb300")
    assert abs(bench.ncu_traffic("a.md", 1000) - 1020) < 1e-9
    assert bench.ncu_traffic("b.md", 1000) is None
    assert bench.ncu_traffic("missing.md", 1000) is None
