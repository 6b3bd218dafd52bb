"""Arithmetic the pages fix about the workloads, checked against the synthetic
shapes and the bench's byte accounting (CPU only, no data generated).

- [LC §6.2] memory table: the KV cache of InternLM2.5-7B-Chat-1M takes 0.5,
  4.29, 8.58, 17.1 and 68.7 GB at 4K, 32K, 64K, 128K and 512K tokens, i.e. 128 KiB per token
  over the model: 32 layers x 8 KV heads x d 128 x fp16 x (K + V) = 4 KiB per
  token and layer, the GQA shape of every workload here.
- [LC §5.3 vs §5.1]: 16K attended tokens = 96 selected blocks x 128 + a 4096
  token Local window.
"""
import numpy as np

import synth

import bench


def _shape_only(params, seq_lens, num_kv_heads=8):
    """A Workload with the shapes of a real one and no pool data."""
    empty = np.empty((0, num_kv_heads, 128, 128), dtype=np.uint16)
    return synth.Workload(name="shape", seed=0, k_pool=empty, v_pool=empty,
                          block_table=np.zeros((len(seq_lens), 1), dtype=np.int32),
                          seq_lens=np.asarray(seq_lens, dtype=np.int32),
                          q=np.empty((len(seq_lens), params.num_q_heads, 128), dtype=np.uint16),
                          params=params)


def test_kv_bytes_per_token_and_the_memory_table():
    per_token_layer = 2 * 8 * 128 * 2          # K and V, 8 KV heads, d 128, fp16
    assert per_token_layer == 4 * 1024
    per_token_model = 32 * per_token_layer      # 32 layers
    assert per_token_model == 128 * 1024
    # the table's GB values are truncated (17.18 GB -> 17.1, 8.589 GB -> 8.58)
    for tokens, gb, places in ((4096, 0.5, 1), (32768, 4.29, 2), (65536, 8.58, 2),
                               (131072, 17.1, 1), (524288, 68.7, 1)):
        assert int(tokens * per_token_model / 10 ** (9 - places)) == round(gb * 10 ** places)
    # dense decode of one 128K layer reads exactly that much K and V
    p = synth.Params(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=10 ** 6,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SHARED)
    assert bench.step_bytes(_shape_only(p, [131072]))["kv"] == 131072 * per_token_layer


def test_sixteen_k_attended_tokens():
    # 96 selected blocks + Local 4096 tokens = 16K attended tokens (no Initial block here)
    p = synth.Params(num_q_heads=32, initial_blocks=0, local_blocks=32, top_k=96,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SHARED)
    kv = bench.step_bytes(_shape_only(p, [131072]))["kv"]
    assert kv // (4 * 1024) == 96 * 128 + 4096 == 16384


def test_step_bytes_of_the_128k_and_1m_workloads():
    # 128K: 991 Context blocks' Quest reps (min + max rows, 8 heads) and the
    # K/V of 1 + 32 + 32 blocks over 8 heads
    p = synth.Params(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=32,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SHARED)
    b = bench.step_bytes(_shape_only(p, [131072]))
    assert b["reps"] == 991 * 8 * 2 * 128 * 2 == 4_059_136
    assert b["kv"] == 65 * 8 * 128 * 128 * 2 * 2 == 34_078_720
    # 1M: 8159 Context blocks; Max reps are half of Quest's
    p1 = synth.Params(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=32,
                      rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE)
    b1 = bench.step_bytes(_shape_only(p1, [1048576]))
    assert b1["reps"] == 8159 * 8 * 2 * 256 and b1["kv"] == b["kv"]
    p1.rep = synth.REP_MAX
    assert bench.step_bytes(_shape_only(p1, [1048576]))["reps"] == b1["reps"] // 2
    # ragged tail: a partial last block counts only its valid tokens
    b2 = bench.step_bytes(_shape_only(p, [131072 - 100]))
    assert b2["kv"] == b["kv"] - 100 * 8 * 128 * 2 * 2
