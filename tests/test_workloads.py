"""The seeded workloads follow their stated recipes: shapes, index structure (distinct entries,
padding layout, recent/uniform split, causal windows), page tables, and the normal generator's
distribution and row-by-row regeneration."""
import numpy as np

from dsa_sparse_attention_mla_gb300 import workloads as W


def _valid_rows(wl):
    return [row[row >= 0] for row in wl.indices]


def test_config1_bf16_direct():
    wl = W.config(1)
    assert (wl.kind, wl.T, wl.H, wl.d_nope, wl.d_rope, wl.d_v) == (0, 17, 64, 256, 0, 256)
    assert wl.num_slots == 8192 and wl.indices.shape == (17, 2112) and wl.sm_scale == 1 / 16
    assert wl.block_table is None
    for row in wl.indices:
        v = row[row >= 0]
        assert v.size == 2051 and np.unique(v).size == 2051 and v.max() < 8192
        assert (row[2051:] == -1).all()  # -1 tail


def test_config2_fp8_paged():
    wl = W.config(2)
    assert (wl.kind, wl.T, wl.d_nope, wl.d_rope, wl.page_size) == (1, 8, 256, 0, 64)
    assert wl.indices.shape == (8, 2048) and (wl.indices >= 0).all()
    assert all(np.unique(r).size == 2048 for r in wl.indices)
    # one request of 16384 positions over a random permutation of 256 pages
    assert np.array_equal(np.sort(wl.block_table.ravel()), np.arange(256))
    assert wl.kv.rows == 16384 and wl.kv.cols == 256


def test_config3_fp8_paged_decode():
    wl = W.config(3)
    assert (wl.kind, wl.T, wl.page_size, wl.sm_scale) == (1, 256, 64, 1 / 16)
    assert wl.num_slots == 256 * 32768 and wl.indices.shape == (256, 2112)
    assert wl.block_table.shape == (256, 512)
    assert np.array_equal(np.sort(wl.block_table.ravel()), np.arange(256 * 512))
    assert np.array_equal(wl.req_of_token, np.arange(256))
    scattered = 0
    for row in wl.indices:
        v = row[row >= 0]
        assert v.size == 2048 and np.unique(v).size == 2048 and v.max() < 32768
        assert (v >= 32768 - 4096).sum() == 1434  # 70% from the last 4096 positions
        if not (row[2048:] == -1).all():
            scattered += 1
    assert scattered == 13  # 5% of the tokens carry their 64 -1 entries inside the list


def test_config4_causal_prefill():
    wl = W.config(4)
    assert (wl.kind, wl.T, wl.num_slots) == (0, 8192, 8192) and wl.indices.shape == (8192, 2048)
    assert int((wl.indices >= 0).sum()) == 14_681_088
    rng = np.random.default_rng(0)
    for t in np.concatenate([[0, 1, 127, 2046, 2047, 2048, 8191], rng.choice(8192, 24, replace=False)]):
        row = wl.indices[t]
        v = row[row >= 0]
        assert (row[v.size:] == -1).all()  # -1 tail
        if t < 2048:
            assert np.array_equal(np.sort(v), np.arange(t + 1))
        else:
            assert v.size == 2048 and np.unique(v).size == 2048 and v.max() == t
            assert np.isin(np.arange(t - 127, t + 1), v).all()  # the last 128 positions
            assert (v <= t - 128).sum() == 1920


def test_config5_control():
    wl = W.config(5)
    assert (wl.kind, wl.T, wl.d_nope, wl.d_rope, wl.d_v, wl.sm_scale) == (1, 1024, 512, 64, 512, 1 / 24)
    assert wl.num_slots == 65536 and wl.kv.cols == 576 and wl.q.cols == 576
    assert wl.indices.shape == (1024, 2048) and (wl.indices >= 0).all()
    assert all(np.unique(r).size == 2048 for r in wl.indices[:64])


def test_normal_rows_distribution_and_regeneration():
    gen = W.config(3).kv
    rows = np.array([0, 5, 1_000_000, gen.rows - 1])
    part = gen.bits(rows)
    again = np.stack([gen.bits(np.array([r]))[0] for r in rows])
    assert np.array_equal(part, again)  # any row is regenerated alone, bit for bit
    x = (gen.bits(np.arange(4096)).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(np.mean(np.abs(x) > 1.96) - 0.05) < 0.005  # two-sided 5% tail of N(0, 1)
