"""Host-side pieces of the benchmark that need no GPU: the launch plan mirrors the
library's grouping, algorithmic traffic counts each weight once, the roofline traffic
figure is withheld when the kernel sources changed."""
import json
import os

import pytest

import bench
from synth import WORKLOADS, weight_bytes


@pytest.mark.parametrize("name,n_inject,n_draft", [
    ("qwen3-8b-b1-ctx2048-B16", 1, 12),          # one 16-row pass; embed, qkv, 5 x (attn, chain)
    ("qwen3-8b-b32-ctx512..8192-B16", 2, 18),    # 512 rows in 256-row passes
    ("llama3.1-8b-L8-b4-ctx32768-B16", 1, 18),   # 64 rows: one pass; 8 layers
])
def test_launch_plan_shape(name, n_inject, n_draft):
    w = WORKLOADS[name]
    plan = bench.launch_plan(w.shape, w.batch, w.block, 4.0, w.ctx)
    assert len(plan["inject"]) == n_inject and len(plan["draft"]) == n_draft and len(plan["verify"]) == 1
    kinds = [k for _, k, _, _ in plan["draft"]]
    assert kinds.count("attn") == w.shape.n_layers


def test_step_bytes_count_each_weight_once():
    w = WORKLOADS["qwen3-8b-b32-ctx512..8192-B16"]
    s = w.shape
    byt, fl = bench.step_bytes_flops(s, w.batch, w.block, w.ctx, 4.0)
    wb = sum(v for k, v in weight_bytes(s).items() if k != "embed_row")
    kv = s.n_layers * bench.attn_bytes_flops(s, w.batch, w.block, w.ctx)[0]
    logits = 4 * w.batch * w.block * s.vocab
    # weights once, K/V once per layer, logits once, plus activation rows (well under 1 GB)
    assert wb + kv + logits < byt < wb + kv + logits + 1e9
    assert fl > 2 * w.batch * w.block * s.hidden * s.vocab * 0.9


def test_traffic_withheld_when_sources_differ(tmp_path, monkeypatch):
    t = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert set(t) >= {"launch", "workload", "traffic_bytes", "sources", "sources_sha256"}
    assert bench.measured_traffic("no-such-launch", t["workload"]) is None
    (tmp_path / "profiles").mkdir()
    t2 = dict(t, sources_sha256="0" * 64)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(t2))
    for src in t["sources"]:
        d = tmp_path / os.path.dirname(src)
        d.mkdir(parents=True, exist_ok=True)
        (tmp_path / src).write_bytes(open(os.path.join(bench.ROOT, src), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic(t["launch"], t["workload"]) is None


def test_reference_and_cuda_arms_print_the_same_config():
    """Both arms describe the workload with one function, so their `config` objects match."""
    w = WORKLOADS["qwen3-8b-b1-ctx2048-B16"]
    c = bench.workload_config(w, 1, 0)
    assert c["workload"] == w.name and c["block"] == 16 and c["ctx"] == 2048 and c["batch_per_gpu"] == 1
    assert "l2" in c and c == bench.workload_config(w, 1, 0)


def test_kv_counted_at_two_bytes_per_element():
    w = WORKLOADS["llama3.1-8b-L8-b4-ctx32768-B16"]
    s = w.shape
    kvb, _ = bench.attn_bytes_flops(s, w.batch, w.block, w.ctx)
    n_kv = (w.ctx + w.block) * s.n_kv_heads * s.head_dim * w.batch
    assert kvb - 6 * w.batch * w.block * s.n_heads * s.head_dim == 4 * n_kv
