"""bench.py's CPU side: the reference arm's JSON line (the fp64 oracle timed
on the host) and the oracle samples behind the cpu_baseline fields."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_fp32", "--steps", "2", "--warmup", "3", "--ref-rows", "16"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_fp32"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_topk_oracle_sample_counts_kept_pairs():
    sys.path.insert(0, ROOT)
    import bench
    import oracle.focus_ref as ref
    from learned_group_sparse_focus_gb300 import synth
    wl = synth.workload("tiny_fp32", n=96, K=4, w=8)
    x = synth.draw(wl)
    flops, secs, desc = bench.oracle_sample_topk(wl, x, 10, [0], seed=3, k=2)
    assert secs > 0 and "top-2" in desc
    # the FLOPs are 4 d per kept pair of the sampled rows, under the top-2 rule
    gid, _ = ref.assign_topk(x["h"], x["W"], x["C"], 2)
    rows = np.sort(np.random.default_rng(3).choice(wl.n, size=10, replace=False))
    kept = int(ref.keep_mask_rows_topk(gid[0, 0], wl.w, rows).sum())
    assert flops == 4 * wl.d * kept


def test_traffic_record_only_for_its_workload_and_source(tmp_path):
    sys.path.insert(0, ROOT)
    import hashlib
    import json
    import bench
    src = os.path.join(ROOT, "learned_group_sparse_focus_gb300", "csrc", "attn_tc.cu")
    sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
    rec = {"bytes_per_launch": 123, "workload": "gqa_32k", "source": "attn_tc.cu", "source_sha1": sha}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"attn_tc_group_pass": rec,
                                "attn_tc_local_pass": dict(rec, source_sha1="0" * 40)}))
    got = bench.traffic_record("attn_tc_group_pass", "gqa_32k", str(path))
    assert got is not None and got["bytes_per_launch"] == 123
    assert bench.traffic_record("attn_tc_group_pass", "llama7b_8k", str(path)) is None   # other workload
    assert bench.traffic_record("attn_tc_local_pass", "gqa_32k", str(path)) is None      # source changed
    assert bench.traffic_record("no_such_kernel", "gqa_32k", str(path)) is None


def test_layer_launch_count_follows_the_index_form():
    # the index build is two launches for problems of at most 4,096 items and
    # 256 groups (one block per problem, then the work list), five otherwise
    sys.path.insert(0, ROOT)
    import bench
    assert bench.index_launches(256, 4) == 2
    assert bench.index_launches(4096, 256) == 2
    assert bench.index_launches(4097, 16) == 5
    assert bench.index_launches(1024, 257) == 5
    assert bench.index_launches(32768, 64) == 5
