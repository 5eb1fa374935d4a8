"""The compact sub-problem the full-size GPU tests hand to the oracle (only the slots the sampled
tokens name, packed by the oracle from the seeded source rows, indices remapped through the
page table) gives the same result as the oracle over the whole cache."""
import numpy as np

from dsa_sparse_attention_mla_gb300 import workloads as W

from _helpers import oracle_cache, run_oracle
from test_gpu_fullsize import _oracle_tokens


def test_compact_subproblem_equals_full_oracle_paged_fp8():
    wl = W.fp8_paged(T=6, requests=3, positions=1024, page_size=64, topk=160, n_valid=150, seed=71,
                     sm_scale=1 / 16, scatter_frac=0.5)
    if wl.kv_slot is not None:  # the compact view assumes slot i holds source row i
        wl.kv_slot = None
    tokens = np.array([0, 2, 5])
    full, full_lse, bad = run_oracle(wl, oracle_cache(wl), tokens=tokens)
    assert bad == 0
    out, lse, rounded = _oracle_tokens(wl, tokens)
    np.testing.assert_array_equal(out, full)
    np.testing.assert_array_equal(lse, full_lse)
    assert rounded is not None


def test_compact_subproblem_equals_full_oracle_bf16_direct():
    wl = W.bf16_direct(T=4, slots=700, topk=96, n_valid=90, seed=72, sm_scale=1 / 16)
    tokens = np.array([1, 3])
    full, full_lse, _ = run_oracle(wl, oracle_cache(wl), tokens=tokens)
    out, lse, rounded = _oracle_tokens(wl, tokens)
    np.testing.assert_array_equal(out, full)
    np.testing.assert_array_equal(lse, full_lse)
    assert rounded is None
