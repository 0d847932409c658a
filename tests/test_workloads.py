"""The synthetic workloads against the shapes the pages print (CPU only)."""
import numpy as np

import synth


def _golden():
    out = {}
    with open(__file__.replace("test_workloads.py", "golden/llama_cpp_090_pr_benchmark_shape.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                out[k] = int(v)
    return out


def test_golden_shape_is_self_consistent():
    g = _golden()
    assert g["parallel_sequences"] * g["prompt_tokens_per_sequence"] == g["total_prompt_tokens"]
    assert g["parallel_sequences"] * g["generated_tokens_per_sequence"] == g["total_generated_tokens"]
    assert g["total_prompt_tokens"] <= g["context_capacity"]


def test_prefill_run_layout_matches_the_printed_benchmark_shape():
    g = _golden()
    rows = synth.prefill_runs_layout(g["parallel_sequences"], g["prompt_tokens_per_sequence"], g["ubatch"])
    assert rows.shape == (4, 99936)
    flat = rows.ravel()
    assert len(np.unique(flat)) == flat.size                 # no pool row is shared
    assert flat.min() == 0 and flat.max() == g["total_prompt_tokens"] - 1 < g["context_capacity"]
    # each ubatch-sized run is contiguous in the pool
    for s in range(4):
        d = np.diff(rows[s])
        breaks = np.nonzero(d != 1)[0]
        assert np.all((breaks + 1) % g["ubatch"] == 0)


def test_small_workloads_have_the_stated_structure():
    p = synth.decode_fp16_small()
    assert p.q.shape == (2, 1, 8, 128) and p.k.shape == (4096, 2, 128) and p.L == 1024
    assert [(p.kv_rows[s] >= 0).sum() for s in range(2)] == [1000, 1000]
    assert len(set(p.kv_rows[p.kv_rows >= 0].tolist())) == 2000
    sp = synth.sparse_bf16()
    r = sp.kv_rows[0]
    assert r.size == 2048 and np.all(np.diff(r) > 0)
    assert r[:4].tolist() == [0, 1, 2, 3] and r[-512:].tolist() == list(range(262144 - 512, 262144))


def test_paged_workload_page_table_is_a_permutation():
    p = synth.paged_int8(n_seq=8, lo=100, hi=3000)
    pages = p.page_table[p.page_table >= 0]
    assert sorted(pages.tolist()) == list(range(p.R // 64))
    assert np.all(p.seq_len >= 100) and np.all(p.seq_len <= 3000)
    assert p.L == p.page_table.shape[1] * 64
