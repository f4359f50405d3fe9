"""The block manager under decoding-like churn (CPU): parallel sampling and a
beam-search-like fork/free loop through the C++ manager; the memory saved by
sharing grows with the number of sequences sharing a prompt, and every block
returns to the free list at the end (checked inside the run)."""
import bench


def test_sharing_savings_synthetic():
    r = bench.sharing_savings(seed=7)
    ps, bs = r["parallel_sampling"], r["beam_search"]
    assert 0 < ps[2] < ps[4] < ps[6] < 1
    assert 0 < bs[4] < bs[8] < 1
