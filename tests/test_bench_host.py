"""Host-side pieces of bench.py (no GPU): the ncu-summary lookup that feeds
roofline.traffic, the algorithmic byte counts and the paged workload's
lengths."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import kvq_inputs as ki  # noqa: E402


def _recorded_sha(name):
    for line in open(os.path.join(ROOT, "profiles", name)):
        if line.startswith("source_sha"):
            return line.split("=", 1)[1].strip()
    return None


def test_committed_profiles_parse_and_guard_on_source_hash():
    # the figure is returned only for the sources the summary was captured on
    sha = _recorded_sha("decode_tc_kernel_mha7b.txt")
    assert sha and len(sha) == 16
    t = bench.profile_traffic("decode_tc_kernel_mha7b.txt", sha)
    assert t is not None
    # DRAM traffic of the captured launch is the algorithmic bytes within 1%
    alg = bench.decode_alg_bytes(ki.WORKLOADS["mha7b"], ki.WORKLOADS["mha7b"].T + 1)
    assert abs(t - alg) / alg < 0.01
    assert bench.profile_traffic("decode_tc_kernel_mha7b.txt", "0" * 16) is None   # stale counters: no figure
    assert bench.profile_traffic("no_such_summary.txt", sha) is None


def test_algorithmic_bytes_match_the_per_token_table():
    # per token and kv head, D = 128: INT4/Gv64/Bk64 + 1% outliers = 152 B; INT3/Gv32/Bk128 = 124 B; INT2 = 92 B
    for name, per_tok in (("gqa8b", 152), ("int3", 124), ("int2", 92)):
        w = ki.WORKLOADS[name]
        qo = 2 * w.B * w.H_q * w.D * 2
        assert bench.decode_alg_bytes(w, w.T) == w.B * w.H_kv * w.T * per_tok + qo
    w = ki.WORKLOADS["mha7b"]                      # no outliers: 144 B
    assert bench.decode_alg_bytes(w, w.T) == w.B * w.H_kv * w.T * 144 + 2 * w.B * w.H_q * w.D * 2


def test_paged_lengths_are_ragged_whole_blocks():
    for name in ("gqa8b", "mha7b", "int3"):
        w = ki.WORKLOADS[name]
        lens = bench.paged_lengths(w)
        assert len(lens) == w.B and lens[0] == w.T
        assert all(L % w.key_block == 0 and L >= w.key_block for L in lens)
        assert all(a > b for a, b in zip(lens, lens[1:]))
